"""The multi-rank host logic of the benchmark on CPU: two `gloo` ranks on
127.0.0.1.  Under torchrun every rank quantizes and multiplies its own batch
of tokens (weak scaling, no collective on the data path); the only
collectives are the timing's max-over-ranks and the barriers.  These tests
check that each rank draws its own batch (rank 0 the workload's own), that
the reduction returns the slowest rank's time on every rank, and the
whole-job rate that follows from it."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    import synth

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.WORKLOADS["tiny"]
        seed = bench.rank_seed(w.seed, rank)
        batch = synth.make_inputs("tiny", seed=seed)["A"]
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(local_ms, dist, "cpu")
        rate = bench.whole_job_rate(100.0, world, 4, slowest)
        np.save(os.path.join(out_dir, f"batch{rank}.npy"), batch)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as fh:
            fh.write(f"{seed} {slowest} {rate}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    import sys
    sys.path.insert(0, ROOT)
    import synth

    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    seeds = [int(r[0]) for r in rows]
    assert seeds[0] == synth.WORKLOADS["tiny"].seed and seeds[1] != seeds[0]
    for r in rows:
        assert float(r[1]) == 15.0                    # the slowest rank's time, on every rank
        assert float(r[2]) == pytest.approx(2 * 100.0 * 4 / 15e-3)
    b0 = np.load(tmp_path / "batch0.npy")
    b1 = np.load(tmp_path / "batch1.npy")
    assert np.array_equal(b0, synth.make_inputs("tiny")["A"])  # rank 0: the workload's batch
    assert b0.shape == b1.shape and not np.array_equal(b0, b1)  # rank 1: its own batch


def test_single_process_needs_no_collective():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(10.0, 1, 2, 1000.0) == pytest.approx(20.0)

"""Two host threads calling the library at once, each on its own CUDA stream
(the C ABI allows it): both get correct results.  The GEMM tile used here is
not used by the test files collected before this one, so both threads reach
its first-use set-up together."""
import threading

import numpy as np
import pytest
import torch

import synth
from tests._helpers import assert_codes_equal, assert_gemm_f32, dev, dev_bf16, host

pytestmark = pytest.mark.gpu

BLOCK = 0
TILE_256x160_PAIR = 3


def test_two_threads_two_streams(fp8bs, oracle_mod):
    cases = []
    for seed in (1, 2):
        rng = np.random.default_rng(seed)
        a_bits, _ = synth.normal_with_outlier_columns(rng, (384, 1024), 3, 50.0)
        w_bits = synth.normal(rng, (640, 1024), 0.02)
        a, sa = oracle_mod.quant_act_1x128(a_bits)
        b, sb = oracle_mod.quant_weight_128x128(w_bits)
        cases.append({"x": dev_bf16(a_bits), "q_ref": a, "a": dev(a), "sa": dev(sa), "b": dev(b),
                      "sb": dev(sb), "ref": oracle_mod.gemm(a, sa, b, sb, BLOCK)})
    torch.cuda.synchronize()
    start = threading.Barrier(2)
    errors = []

    def work(case):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                start.wait()
                for _ in range(5):
                    case["q"], _ = fp8bs.quant_act_1x128(case["x"])
                    case["c"] = fp8bs.gemm(case["a"], case["sa"], case["b"], case["sb"], BLOCK,
                                           out_dtype=torch.float32, tile=TILE_256x160_PAIR)
            stream.synchronize()
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(c,)) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for i, case in enumerate(cases):
        assert_codes_equal(case["q"], case["q_ref"], f"thread {i} codes")
        assert_gemm_f32(host(case["c"]), case["ref"], f"thread {i} gemm")
    assert fp8bs.get_device_error(torch.device("cuda", 0)) == fp8bs.OK

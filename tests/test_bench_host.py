"""Host-side logic of the bench.  The clock sampler, run on the CPU against a
fake nvidia-smi, must be sampling before the timed region starts, keep only
the samples taken while the region ran, and report the throttle reasons it
saw.  The algorithmic byte counts match the per-element figures."""
import os
import stat
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FAKE = """#!/bin/sh
# prints one sample line every 10 ms: SM MHz, max MHz, event-reason bits
i=0
while true; do
  if [ -f "$FAKE_SMI_FLAG" ]; then echo "1500, 2032, 0x0000000000000004"; else echo "2032, 2032, 0x0000000000000000"; fi
  i=$((i+1))
  sleep 0.01
done
"""


@pytest.fixture
def fake_smi(tmp_path, monkeypatch):
    exe = tmp_path / "nvidia-smi"
    exe.write_text(FAKE)
    exe.chmod(exe.stat().st_mode | stat.S_IEXEC)
    flag = tmp_path / "capped"
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    monkeypatch.setenv("FAKE_SMI_FLAG", str(flag))
    sys.path.insert(0, ROOT)
    import bench
    return bench, flag


def _sampler(bench):
    s = bench.ClockSampler(0)
    s.mode = "smi"  # no NVML on this host path
    return s


def test_sampler_records_region(fake_smi):
    bench, _ = fake_smi
    s = _sampler(bench)
    with s:
        assert s.lines, "sampling must have started before the region"
        time.sleep(0.2)
    out = s.summary()
    assert out["samples"] >= 5
    assert out["sm_mhz"] == 2032.0 and out["sm_max_mhz"] == 2032.0
    assert out["reasons"] == []


def test_sampler_reports_reasons_inside_region_only(fake_smi):
    bench, flag = fake_smi
    s = _sampler(bench)
    with s:
        flag.write_text("1")
        time.sleep(0.2)
    flag.unlink()
    out = s.summary()
    assert "sw_power_cap" in out["reasons"]
    assert out["sm_mhz"] == 1500.0


def test_algorithmic_bytes_per_element():
    """The bench's byte counts are the per-element figures the roofline
    uses: Q1 2 + 1 + 4/128, Q2 3 + 4/16384 (4 + 8/16384 with the transposed
    copy), the dual quantizer 2 + 2 * (1 + 4/128), Q3 2 * (1 + 4/128)."""
    sys.path.insert(0, ROOT)
    import bench
    M, K = 4096, 7168
    n = M * K
    assert bench.algorithmic_bytes_q1(M, K) / n == pytest.approx(3 + 4 / 128)
    assert bench.algorithmic_bytes_q2(M, K) / n == pytest.approx(3 + 4 / 16384)
    assert bench.algorithmic_bytes_q2(M, K, transposed=True) / n == pytest.approx(4 + 8 / 16384)
    assert bench.algorithmic_bytes_dual(M, K) / n == pytest.approx(2 + 2 * (1 + 4 / 128))
    assert bench.algorithmic_bytes_q3(M, K) / n == pytest.approx(2 * (1 + 4 / 128))


def test_cpu_legs_sample_whole_b_blocks():
    """The CPU legs quantize B in 128x128 blocks on a sample of its rows:
    every sample starts on a block boundary and stays inside B, so the
    sample's blocks are blocks of the full-size quantization."""
    sys.path.insert(0, ROOT)
    import bench
    N, n_s = 8192, 256
    for r0 in list(range(0, N, 37)) + [N - 1, N - 8, 0]:
        b0 = bench._b_rows(N, r0, n_s)
        assert b0 % 128 == 0 and 0 <= b0 and b0 + n_s <= N, (r0, b0)

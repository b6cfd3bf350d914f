"""The quantizer kernels replace the IEEE division x / s by a correctly
rounded reciprocal and Markstein correction steps (one step for bf16
inputs, two for FP32 inputs).  Their bit-exactness against the oracle's
division rests on the claim that this gives the same code as fl32(x / s)
for every input the fast path sees.  These CPU tests check that claim with
a small C program (tests/quotient_check.c) that restates the kernels'
arithmetic with fmaf:

- one step, E4M3: every positive finite bf16 max-abs value whose scale
  fl32(amax / 448) is at least 2^-92 (the kernels send smaller scales to the
  exact division) against every bf16 x with |x| <= amax, both signs
  (about 10^9 pairs);
- one step, E5M6 cache: the same with 65024 in place of 448;
- two steps, FP32 inputs (the re-tiling and the epilogue quantizer): a
  seeded sample of 20 million pairs;
- the planted mistake (the product without its correction step) must be
  caught.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "quotient_check.c")


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path_factory.mktemp("quotient") / "quotient_check")
    flags = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp"]
    with open("/proc/cpuinfo") as fh:
        if " fma " in fh.read():
            flags.append("-mfma")  # hardware fmaf; libm's software fmaf is also exact
    subprocess.run([gcc, *flags, "-o", exe, SRC, "-lm"], check=True)
    return exe


def _run(exe, *args):
    out = subprocess.run([exe, *args], check=True, capture_output=True, text=True,
                         timeout=600).stdout
    last = out.strip().splitlines()[-1]
    fields = dict(kv.split("=") for kv in last.split())
    return int(fields["pairs"]), int(fields["mismatches"]), out


def test_one_step_e4m3_every_bf16_pair(checker):
    pairs, bad, out = _run(checker, "one_step_e4m3")
    assert pairs > 1_000_000_000 and bad == 0, out


def test_one_step_e5m6_every_bf16_pair(checker):
    pairs, bad, out = _run(checker, "one_step_e5m6")
    assert pairs > 1_000_000_000 and bad == 0, out


def test_two_step_fp32_sample(checker):
    pairs, bad, out = _run(checker, "two_step", "20000000")
    assert pairs >= 19_000_000 and bad == 0, out


def test_check_catches_a_missing_correction(checker):
    pairs, bad, _ = _run(checker, "no_step_e4m3")
    assert pairs > 1_000_000_000 and bad > 1000

"""The E5M6 cache kernels encode and decode 12-bit codes by bit arithmetic:
the fast encoder rounds and rebiases a negated quotient's FP32 pattern with
one integer addition and makes the subnormal multiple of 2^-20 with one
fused multiply-add; the exact-division path has its own encoder; the decoder
shifts two codes into an IEEE f16x2 word and converts it; eight codes are
packed into three little-endian words.  The GPU parity tests compare these
with the oracle on the inputs they draw; these CPU tests check them on every
input (tests/e5m6_codec_check.c restates the kernels' operations and
compares them with the format's definition computed in double precision):

- the fast encoder on every FP32 pattern with |q| below 65280 (the largest
  finite code 65024 and the midpoint above it; a group's quotient stays
  within 65024 (1 + 2^-23)), both signs;
- the exact-division encoder on all 2^32 FP32 patterns (NaN, Inf,
  saturation, subnormals, both zeros);
- the decoder for every code at each position of a 48-bit group;
- the packer on a seeded sample;
- the planted mistake (the rounding increment dropped) must be caught.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "e5m6_codec_check.c")


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path_factory.mktemp("e5m6") / "e5m6_codec_check")
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


def test_fast_encoder_every_quotient(checker):
    pairs, bad, out = _run(checker, "fast")
    assert pairs == 2 * 0x477F0000 and bad == 0, out


def test_general_encoder_every_fp32(checker):
    pairs, bad, out = _run(checker, "general")
    assert pairs == 1 << 32 and bad == 0, out


def test_decoder_every_code_every_position(checker):
    pairs, bad, out = _run(checker, "decode")
    assert pairs == 4 * 16 * 4096 * 4 and bad == 0, out


def test_packer_sample(checker):
    pairs, bad, out = _run(checker, "pack", "1000000")
    assert pairs == 8_000_000 and bad == 0, out


def test_check_catches_a_missing_rounding_increment(checker):
    pairs, bad, _ = _run(checker, "fast_nocarry")
    assert pairs == 2 * 0x477F0000 and bad > 1000

"""The affine encoder computes each code from RN((w - b) / s) without a division per weight:
u = RN(d yk + RN(d yek)) with y = RN(1/s), e0 = 1 - s y, yek = RN(y e0)/K, yk = y/K.  This checks,
on the CPU in plain C, that the identity u K = RN(d / s) holds for every bf16 significand of s and
every binary32 d in [2^-4, 2^7) (a quotient's rounding depends on d and s only through their
significands and the exponent difference), and on a sample at the ends of the exponent range the
encoder uses unscaled.  The GPU parity tests compare the encoder's codes with the oracle's
division bit for bit; this covers the ties and near-ties that random weights almost never hit."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_division_free_quotient_is_correctly_rounded():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "quotient_check")
        subprocess.check_call([gcc, "-O2", "-fno-fast-math", "-ffp-contract=off", "-pthread",
                               os.path.join(HERE, "quotient_check.c"), "-o", exe, "-lm"])
        r = subprocess.run([exe, "97"], capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("0 mismatches"), r.stdout

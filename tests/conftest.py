import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Acceptance bound for every floating-point output of the path:
#   |y - y_ref| <= REL * absref + ABS, absref = sum of |w*x| terms from the fp64 oracle.
REL = 1e-3
ABS = 1e-6


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def assert_within_bound(y, y_ref, absref, rel=REL, abs_=ABS, what="y"):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    absref = np.asarray(absref, dtype=np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs"
    err = np.abs(y - y_ref)
    lim = rel * absref + abs_
    bad = np.nonzero(err > lim)
    if bad[0].size:
        i = tuple(b[0] for b in bad)
        ratio = float(np.max(err / lim))
        raise AssertionError(f"{what}: {bad[0].size} elements out of bound; first at {i}: got {y[i]!r} "
                             f"ref {y_ref[i]!r} err {err[i]:.3e} lim {lim[i]:.3e}; worst err/lim {ratio:.3f}")
    return float(np.max(err / lim)) if err.size else 0.0


@pytest.fixture(scope="session")
def qg():
    """The CUDA library binding, built in-tree first.  GPU tests only."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_int4_affine_gb300 import build

    build.build()
    from moe_int4_affine_gb300 import qg as _qg

    return _qg

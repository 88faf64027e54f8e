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


# host threads for the oracle on full-size checks (ctypes releases the GIL in each C call)
ORACLE_THREADS = max(1, min(32, os.cpu_count() or 1))


def swiglu_bound(g, u, dg, du):
    """Bound on |h~ - h| for h = silu(g) u when |g~ - g| <= dg and |u~ - u| <= du (all float64 arrays).

    h~ - h = silu'(g) u dg' + silu(g~) du' + (silu(g~) - silu(g) - silu'(g) dg') u with |dg'| <= dg,
    |du'| <= du.  |silu''| <= 1/2 everywhere (its maximum is at 0: 2 sigma'(0) = 1/2), so the last
    term is at most |u| dg^2 / 4, and |silu(g~)| <= |silu(g)| + 1.1 dg (|silu'| <= 1.1).  The fp32
    evaluation of h~ from g~ and u~ (expf, a division and two products) adds at most 2^-21 |h|."""
    s = 1.0 / (1.0 + np.exp(-g))
    silu = g * s
    dsilu = s * (1.0 + g * (1.0 - s))
    return (np.abs(dsilu * u) * dg + (np.abs(silu) + 1.1 * dg) * du + 0.25 * np.abs(u) * dg * dg
            + 2.0 ** -21 * np.abs(silu * u))


def dense_layer_reference(gate, up, down, x, threads=ORACLE_THREADS):
    """The dense decode layer y = W_d (silu(W_g x) * (W_u x)) through the oracle, h kept in fp64,
    and the bound every GPU output must meet when each GEMV stage meets the acceptance bound:

      g~, u~ within 1e-3 A_g + 1e-6 and 1e-3 A_u + 1e-6 (A = sum |w x|, per row)
      |h~ - h| <= dh                                   (swiglu_bound)
      |y~ - W_d h~| <= 1e-3 sum_i |W_d[r][i] h~_i| + 1e-6   (the down GEMV, on the fp32 h~ it reads)
      |W_d (h~ - h)| <= sum_i |W_d[r][i]| dh_i
    so |y~ - y| <= 1e-3 (A_h + A_dh) + 1e-6 + A_dh, with A_h = sum_i |W_d[r][i] h_i| and
    A_dh = sum_i |W_d[r][i]| dh_i.  Returns (y_ref, y_bound, h_ref, h_bound), float64."""
    import oracle

    g, ag = oracle.qgemv(gate["packed"], gate["scales"], gate["biases"], x, threads=threads)
    u, au = oracle.qgemv(up["packed"], up["scales"], up["biases"], x, threads=threads)
    h = oracle.swiglu(g, u)
    dh = swiglu_bound(g, u, REL * ag + ABS, REL * au + ABS)
    y, a_h = oracle.qgemv_f64x(down["packed"], down["scales"], down["biases"], h)
    _, a_dh = oracle.qgemv_f64x(down["packed"], down["scales"], down["biases"], dh)
    return y, REL * (a_h + a_dh) + ABS + a_dh, h, dh


def assert_within(y, y_ref, bound, what="y"):
    """|y - y_ref| <= bound elementwise (a bound derived for the comparison at hand)."""
    y = np.asarray(y, dtype=np.float64)
    assert y.shape == np.shape(y_ref), (y.shape, np.shape(y_ref))
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs"
    err = np.abs(y - y_ref)
    bad = np.nonzero(err > bound)
    if bad[0].size:
        i = tuple(b[0] for b in bad)
        raise AssertionError(f"{what}: {bad[0].size} elements out of bound; first at {i}: got {y[i]!r} "
                             f"ref {y_ref[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")
    return float(np.max(err / bound)) if err.size else 0.0


class Guarded:
    """A device buffer with sentinel-filled guard regions on both sides of the part a call may
    write: `t` is the inner view (16-byte aligned); `intact()` reads both guards back.  A kernel
    writing past either end of an output, a workspace or h is caught even where the values it
    was meant to produce are right."""
    GUARD = 4096  # bytes on each side
    SENTINEL = 0xA5

    def __init__(self, shape, dtype, device="cuda"):
        import torch

        shape = (shape,) if isinstance(shape, int) else tuple(shape)
        n = int(np.prod(shape)) if shape else 1
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        inner = (nbytes + 15) // 16 * 16
        self.raw = torch.full((2 * self.GUARD + inner,), self.SENTINEL, dtype=torch.uint8, device=device)
        self.nbytes = nbytes
        self.t = self.raw[self.GUARD:self.GUARD + nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        import torch

        lo = self.raw[:self.GUARD]
        hi = self.raw[self.GUARD + self.nbytes:]
        return bool(torch.all(lo == self.SENTINEL).item()) and bool(torch.all(hi == self.SENTINEL).item())


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

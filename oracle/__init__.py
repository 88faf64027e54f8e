"""fp64 CPU oracle for the int4 affine dequant-GEMV decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The CUDA library never imports, links or
executes anything here, and this package imports nothing from the CUDA library.

The arithmetic lives in ``qg_oracle.c`` (plain C, double precision, the definitions written
out).  This module compiles it with the host C compiler and marshals numpy arrays into it.
Every function returns float64 results plus the ``absref`` scale (sum of |w*x| terms) that the
acceptance bound ``|y - y_ref| <= 1e-3 * absref + 1e-6`` is stated against.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` (closed forms,
exact rational brute force, the pages' router example); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qg_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libqg_oracle.so")
_lib = None
_lock = threading.Lock()

X_BF16 = 0
X_F32 = 1


def build(force: bool = False) -> str:
    """Compile qg_oracle.c into a shared library (strict IEEE: no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f64.restype = ctypes.c_double
            lib.orc_unpack_rows.argtypes = [P, I64, I64, I64, P]
            lib.orc_unpack_rows.restype = None
            lib.orc_qgemv_rows.argtypes = [P, P, P, I64, I64, I64, P, I, I64, I64, P, P]
            lib.orc_qgemv_rows.restype = I
            lib.orc_qgemv_rows_f64x.argtypes = [P, P, P, I64, I64, I64, P, I64, I64, P, P]
            lib.orc_qgemv_rows_f64x.restype = I
            lib.orc_silu.argtypes = [ctypes.c_double]
            lib.orc_silu.restype = ctypes.c_double
            lib.orc_swiglu.argtypes = [P, P, I64, P]
            lib.orc_swiglu.restype = None
            lib.orc_router_topk.argtypes = [P, I, I, I, P, P]
            lib.orc_router_topk.restype = I
            lib.orc_chain_residual.argtypes = [P, I, P, P, I64, I64, I64, P, P]
            lib.orc_chain_residual.restype = None
            lib.orc_moe.argtypes = [P] * 9 + [I64, I64, I64, I64, P, P, I, P, P, P, P]
            lib.orc_moe.restype = I
            lib.orc_qgemm_rows.argtypes = [P, P, P, I64, I64, I64, P, I64, I64, I64, P, P]
            lib.orc_qgemm_rows.restype = I
            lib.orc_code2.argtypes = [P, I64, I64, I64]
            lib.orc_code2.restype = ctypes.c_uint
            lib.orc_qgemv2_rows.argtypes = [P, P, P, I64, I64, P, I, I64, I64, P, P]
            lib.orc_qgemv2_rows.restype = I
            lib.orc_qgemv2_rows_f64x.argtypes = [P, P, P, I64, I64, P, I64, I64, P, P]
            lib.orc_qgemv2_rows_f64x.restype = I
            lib.orc_moe2.argtypes = [P] * 9 + [I64, I64, I64, P, P, I, P, P, P, P]
            lib.orc_moe2.restype = I
            lib.orc_bf16_round.argtypes = [ctypes.c_float]
            lib.orc_bf16_round.restype = ctypes.c_uint16
            lib.orc_quantize_rows.argtypes = [P, I, I64, I64, I, I64, I64, P, P, P]
            lib.orc_quantize_rows.restype = I
            lib.orc_rmsnorm.argtypes = [P, I, P, I64, ctypes.c_double, P]
            lib.orc_rmsnorm.restype = I
            lib.orc_gated_rmsnorm.argtypes = [P, P, I, P, I64, I64, ctypes.c_double, P]
            lib.orc_gated_rmsnorm.restype = I
            lib.orc_sigmoid.argtypes = [ctypes.c_double]
            lib.orc_sigmoid.restype = ctypes.c_double
            lib.orc_sigmoid_scalar_fma.argtypes = [ctypes.c_double, P, P, P, I64, P, P]
            lib.orc_sigmoid_scalar_fma.restype = None
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _xtype(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return X_BF16
    if x.dtype == np.float32:
        return X_F32
    raise TypeError(f"x must be bf16 bits (uint16) or float32, got {x.dtype}")


def bf16_to_f64(bits) -> float:
    return _L().orc_bf16_to_f64(int(bits))


def unpack(packed: np.ndarray, in_dim: int, r0: int = 0, r1: int | None = None) -> np.ndarray:
    """Codes q[r][j] (uint8) of rows r0..r1-1 of a [out][in/8] u32 weight."""
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    out = packed.size // (in_dim // 8)
    r1 = out if r1 is None else r1
    q = np.empty((r1 - r0, in_dim), dtype=np.uint8)
    _L().orc_unpack_rows(_p(packed), in_dim, r0, r1, _p(q))
    return q


def qgemv(packed, scales, biases, x, group_size: int = 64, rows=None, threads: int = 1):
    """y, absref (float64) of y = W x for the requested rows (default all).

    ``rows`` is None (all rows) or a (r0, r1) range.  ``threads`` > 1 splits the row range
    over host threads (ctypes releases the GIL for the duration of each C call).
    """
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    biases = np.ascontiguousarray(biases, dtype=np.uint16)
    x = np.ascontiguousarray(x)
    in_dim = x.shape[-1]
    out = packed.size // (in_dim // 8)
    r0, r1 = (0, out) if rows is None else (int(rows[0]), int(rows[1]))
    y = np.empty(r1 - r0, dtype=np.float64)
    a = np.empty(r1 - r0, dtype=np.float64)
    xt = _xtype(x)
    L = _L()

    def part(lo, hi):
        rc = L.orc_qgemv_rows(_p(packed), _p(scales), _p(biases), out, in_dim, group_size, _p(x), xt, lo, hi,
                              ctypes.c_void_p(y.ctypes.data + 8 * (lo - r0)),
                              ctypes.c_void_p(a.ctypes.data + 8 * (lo - r0)))
        if rc != 0:
            raise ValueError(f"orc_qgemv_rows rejected the shape (rc={rc})")

    _split(r0, r1, threads, part)
    return y, a


def qgemv_f64x(packed, scales, biases, x64: np.ndarray, group_size: int = 64):
    """y, absref of W h with h given in float64 (the oracle's own intermediate)."""
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    x64 = np.ascontiguousarray(x64, dtype=np.float64)
    in_dim = x64.shape[-1]
    out = packed.size // (in_dim // 8)
    y = np.empty(out, dtype=np.float64)
    a = np.empty(out, dtype=np.float64)
    rc = _L().orc_qgemv_rows_f64x(_p(packed), _p(np.ascontiguousarray(scales, dtype=np.uint16)),
                                  _p(np.ascontiguousarray(biases, dtype=np.uint16)), out, in_dim, group_size,
                                  _p(x64), 0, out, _p(y), _p(a))
    if rc != 0:
        raise ValueError("orc_qgemv_rows_f64x rejected the shape")
    return y, a


def silu(g: float) -> float:
    return _L().orc_silu(float(g))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    h = np.empty_like(g)
    _L().orc_swiglu(_p(g), _p(u), g.size, _p(h))
    return h


def router_topk(logits: np.ndarray, k: int = 8, renorm: bool = True):
    """(idx uint32[k], p float64[k]) in selection order: (logit desc, index asc)."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    idx = np.empty(k, dtype=np.uint32)
    p = np.empty(k, dtype=np.float64)
    rc = _L().orc_router_topk(_p(logits), logits.size, k, 1 if renorm else 0, _p(idx), _p(p))
    if rc != 0:
        raise ValueError("orc_router_topk rejected the arguments")
    return idx, p


def chain_residual(p: np.ndarray, v: np.ndarray, residual: np.ndarray, rows=None):
    """y = residual + sum_k p[k] * v[k]  (v float32 [K][n], residual bf16 bits [n])."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float32)
    residual = np.ascontiguousarray(residual, dtype=np.uint16)
    K, n = v.shape
    i0, i1 = (0, n) if rows is None else (int(rows[0]), int(rows[1]))
    y = np.empty(i1 - i0, dtype=np.float64)
    a = np.empty(i1 - i0, dtype=np.float64)
    _L().orc_chain_residual(_p(p), K, _p(v), _p(residual), n, i0, i1, _p(y), _p(a))
    return y, a


def moe(gate, up, down, idx, p, x, residual, group_size: int = 64):
    """MoE decode step.  gate/up/down are (packed, scales, biases) tuples of stacked experts:
    gate/up packed [E][inter][hidden/8], down packed [E][hidden][inter/8].
    Returns y, absref (float64 [hidden]) and the invalid-slot flag bits."""
    gq, gs, gb = (np.ascontiguousarray(a) for a in gate)
    uq, us, ub = (np.ascontiguousarray(a) for a in up)
    dq, ds, db = (np.ascontiguousarray(a) for a in down)
    E, inter, hw = gq.shape
    hidden = hw * 8
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    p = np.ascontiguousarray(p, dtype=np.float64)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    residual = np.ascontiguousarray(residual, dtype=np.uint16)
    y = np.empty(hidden, dtype=np.float64)
    a = np.empty(hidden, dtype=np.float64)
    flags = _L().orc_moe(_p(gq), _p(gs), _p(gb), _p(uq), _p(us), _p(ub), _p(dq), _p(ds), _p(db), E, hidden, inter,
                         group_size, _p(idx), _p(p), idx.size, _p(x), _p(residual), _p(y), _p(a))
    if flags < 0:
        raise ValueError("orc_moe rejected the shapes")
    return y, a, flags


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """out = x * gamma / sqrt(mean(x^2) + eps) in float64 (x bf16 bits or float32, gamma bf16 bits)."""
    x = np.ascontiguousarray(x)
    gamma = np.ascontiguousarray(gamma, dtype=np.uint16)
    if gamma.size != x.size:
        raise ValueError("gamma and x differ in length")
    out = np.empty(x.size, dtype=np.float64)
    rc = _L().orc_rmsnorm(_p(x), _xtype(x), _p(gamma), x.size, float(eps), _p(out))
    if rc != 0:
        raise ValueError("orc_rmsnorm rejected the arguments")
    return out


def rmsnorm_qgemv(packed, scales, biases, x, gamma, eps: float, group_size: int = 64):
    """y, absref of W rmsnorm(x): the norm in float64, then the GEMV of the normalised vector."""
    return qgemv_f64x(packed, scales, biases, rmsnorm(x, gamma, eps), group_size)


def gated_rmsnorm(y: np.ndarray, z: np.ndarray, gamma: np.ndarray, eps: float, head_dim: int) -> np.ndarray:
    """out = silu(z) * gamma * y / sqrt(mean over the head of y^2 + eps), heads of head_dim
    consecutive elements, float64 (y, z: bf16 bits or float32, the same type; gamma bf16 bits)."""
    y = np.ascontiguousarray(y)
    z = np.ascontiguousarray(z, dtype=y.dtype)
    gamma = np.ascontiguousarray(gamma, dtype=np.uint16)
    if gamma.size != y.size or z.size != y.size:
        raise ValueError("y, z and gamma differ in length")
    out = np.empty(y.size, dtype=np.float64)
    rc = _L().orc_gated_rmsnorm(_p(y), _p(z), _xtype(y), _p(gamma), y.size, int(head_dim), float(eps), _p(out))
    if rc != 0:
        raise ValueError("orc_gated_rmsnorm rejected the arguments")
    return out


def gated_rmsnorm_qgemv(packed, scales, biases, y, z, gamma, eps: float, head_dim: int, group_size: int = 64):
    """out, absref of W gated_rmsnorm(y, z): the norm in float64, then the GEMV of the result."""
    return qgemv_f64x(packed, scales, biases, gated_rmsnorm(y, z, gamma, eps, head_dim), group_size)


def code2(packed, in_dim: int, row: int, j: int) -> int:
    """2-bit code of element j of row `row` (16 per u32, low first)."""
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    return int(_L().orc_code2(_p(packed), in_dim, row, j))


def qgemv2(packed, scales, biases, x, rows=None, threads: int = 1):
    """y, absref of the 2-bit affine GEMV (packed uint32 [out][in/16]); ``threads`` as qgemv."""
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    biases = np.ascontiguousarray(biases, dtype=np.uint16)
    x = np.ascontiguousarray(x)
    in_dim = x.shape[-1]
    out = packed.size // (in_dim // 16)
    r0, r1 = (0, out) if rows is None else (int(rows[0]), int(rows[1]))
    y = np.empty(r1 - r0, dtype=np.float64)
    a = np.empty(r1 - r0, dtype=np.float64)
    xt = _xtype(x)
    L = _L()

    def part(lo, hi):
        rc = L.orc_qgemv2_rows(_p(packed), _p(scales), _p(biases), out, in_dim, _p(x), xt, lo, hi,
                               ctypes.c_void_p(y.ctypes.data + 8 * (lo - r0)),
                               ctypes.c_void_p(a.ctypes.data + 8 * (lo - r0)))
        if rc != 0:
            raise ValueError("orc_qgemv2_rows rejected the shape")

    _split(r0, r1, threads, part)
    return y, a


def qgemv2_f64x(packed, scales, biases, x64: np.ndarray):
    """y, absref of the 2-bit GEMV of an input given in float64 (the 2-bit MoE down's h)."""
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    x64 = np.ascontiguousarray(x64, dtype=np.float64)
    in_dim = x64.shape[-1]
    out = packed.size // (in_dim // 16)
    y = np.empty(out, dtype=np.float64)
    a = np.empty(out, dtype=np.float64)
    rc = _L().orc_qgemv2_rows_f64x(_p(packed), _p(np.ascontiguousarray(scales, dtype=np.uint16)),
                                   _p(np.ascontiguousarray(biases, dtype=np.uint16)), out, in_dim, _p(x64), 0, out,
                                   _p(y), _p(a))
    if rc != 0:
        raise ValueError("orc_qgemv2_rows_f64x rejected the shape")
    return y, a


def moe2(gate, up, down, idx, p, x, residual):
    """The MoE decode step with 2-bit experts (gate/up packed [E][inter][hidden/16], down
    [E][hidden][inter/16]); returns y, absref and the invalid-slot flag bits, as moe()."""
    gq, gs, gb = (np.ascontiguousarray(a) for a in gate)
    uq, us, ub = (np.ascontiguousarray(a) for a in up)
    dq, ds, db = (np.ascontiguousarray(a) for a in down)
    E, inter, hw = gq.shape
    hidden = hw * 16
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    p = np.ascontiguousarray(p, dtype=np.float64)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    residual = np.ascontiguousarray(residual, dtype=np.uint16)
    y = np.empty(hidden, dtype=np.float64)
    a = np.empty(hidden, dtype=np.float64)
    flags = _L().orc_moe2(_p(gq), _p(gs), _p(gb), _p(uq), _p(us), _p(ub), _p(dq), _p(ds), _p(db), E, hidden, inter,
                          _p(idx), _p(p), idx.size, _p(x), _p(residual), _p(y), _p(a))
    if flags < 0:
        raise ValueError("orc_moe2 rejected the shapes")
    return y, a, flags


def bf16_round(f: float) -> int:
    """bf16 bits of a binary32 value, round to nearest, ties to even."""
    return int(_L().orc_bf16_round(float(f)))


def quantize(w: np.ndarray, bits: int = 4, rows=None):
    """Affine group-64 encode of w (bf16 bits or float32, [out][in]): (packed uint32
    [out][in*bits/32], scales bf16 bits [out][in/64], biases bf16 bits [out][in/64])."""
    w = np.ascontiguousarray(w)
    out, in_dim = w.shape
    r0, r1 = (0, out) if rows is None else (int(rows[0]), int(rows[1]))
    packed = np.zeros((out, in_dim * bits // 32), dtype=np.uint32)
    scales = np.zeros((out, in_dim // 64), dtype=np.uint16)
    biases = np.zeros((out, in_dim // 64), dtype=np.uint16)
    rc = _L().orc_quantize_rows(_p(w), _xtype(w), out, in_dim, bits, r0, r1, _p(packed), _p(scales), _p(biases))
    if rc != 0:
        raise ValueError("orc_quantize_rows rejected the arguments")
    return packed[r0:r1], scales[r0:r1], biases[r0:r1]


def sigmoid(g: float) -> float:
    return _L().orc_sigmoid(float(g))


def sigmoid_scalar_fma(gate: float, value: np.ndarray, base: np.ndarray, residual=None):
    """out = base + sigmoid(gate) * value (+ residual bf16 bits), and absref."""
    value = np.ascontiguousarray(value, dtype=np.float32)
    base = np.ascontiguousarray(base, dtype=np.float32)
    if residual is not None:
        residual = np.ascontiguousarray(residual, dtype=np.uint16)
    n = value.size
    out = np.empty(n, dtype=np.float64)
    a = np.empty(n, dtype=np.float64)
    _L().orc_sigmoid_scalar_fma(float(gate), _p(value), _p(base), None if residual is None else _p(residual), n,
                                _p(out), _p(a))
    return out, a


def qgemm(packed, scales, biases, X, group_size: int = 64, rows=None, threads: int = 1):
    """Y[t][r] (float64 [T][r1-r0]) and absref for bf16 X [T][in]."""
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    X = np.ascontiguousarray(X, dtype=np.uint16)
    T, in_dim = X.shape
    out = packed.size // (in_dim // 8)
    r0, r1 = (0, out) if rows is None else (int(rows[0]), int(rows[1]))
    if threads <= 1:
        Y = np.empty((T, r1 - r0), dtype=np.float64)
        A = np.empty((T, r1 - r0), dtype=np.float64)
        rc = _L().orc_qgemm_rows(_p(packed), _p(np.ascontiguousarray(scales, dtype=np.uint16)),
                                 _p(np.ascontiguousarray(biases, dtype=np.uint16)), out, in_dim, group_size, _p(X), T,
                                 r0, r1, _p(Y), _p(A))
        if rc != 0:
            raise ValueError("orc_qgemm_rows rejected the shape")
        return Y, A
    Ys, As = [], []
    for t in range(T):
        y, a = qgemv(packed, scales, biases, X[t], group_size, (r0, r1), threads)
        Ys.append(y)
        As.append(a)
    return np.stack(Ys), np.stack(As)


def _split(r0: int, r1: int, threads: int, fn) -> None:
    n = r1 - r0
    if threads <= 1 or n < 2 * threads:
        fn(r0, r1)
        return
    step = (n + threads - 1) // threads
    bounds = [(lo, min(lo + step, r1)) for lo in range(r0, r1, step)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for f in [ex.submit(fn, lo, hi) for lo, hi in bounds]:
            f.result()

"""ctypes binding of libqg (include/qg.h): the same entry points, argument marshalling only.

Tensors are torch CUDA tensors (torch supplies device memory and streams); the binding passes
their data pointers and the current CUDA stream to the C ABI and raises QGError on a non-zero
return code.  Importing this module raises ImportError when the compiled library is missing: no
call can fall back to anything else.  Build it with ``python -m moe_int4_affine_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libqg.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"libqg.so not built ({LIB_PATH}); run `python -m moe_int4_affine_gb300.build`")
lib = ctypes.CDLL(LIB_PATH)

# ---------------------------------------------------------------- constants (include/qg.h)
QG_OK, QG_EINVAL, QG_EALIGN, QG_EWORKSPACE, QG_ELAUNCH, QG_ENOTSUP, QG_EDEVICE = 0, -1, -2, -3, -4, -5, -6
QG_STATUS_BAD_EXPERT, QG_STATUS_TIMEOUT = 1, 2
QG_X_BF16, QG_X_F32 = 0, 1
QG_EPI_NONE, QG_EPI_SWIGLU = 0, 1
QG_OP_QGEMV, QG_OP_MULTI, QG_OP_MOE, QG_OP_QGEMM, QG_OP_LAYER, QG_OP_LAYER_HOST, QG_OP_MOE_PREFILL, QG_OP_GATED_NORM = 0, 1, 2, 3, 4, 5, 6, 7
QG_NOALLOC_MOE_MAX_FLOATS = 32768


class qg_int4_weight(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p),
                ("out", ctypes.c_int32), ("in_", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("n_mat", ctypes.c_int32)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_W = ctypes.POINTER(qg_int4_weight)
lib.qgemv_int4.argtypes = [_W, _P, _I, _P, _P]
lib.qgemv_int4_multi.argtypes = [_I, _W, _P, _I, ctypes.POINTER(_P), _I, _P]
lib.moe_router_topk.argtypes = [_P, _I, _I, _I, _P, _P, _P]
lib.moe_gather_qgemv_int4.argtypes = [_W, _W, _W, _P, _P, _I, _P, _P, _P, _P, ctypes.c_size_t, _P]
lib.moe_layer_int4.argtypes = [_P, _I, _W, _W, _W, _I, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
lib.moe_prefill_int4.argtypes = [_P, _I, _I, _W, _W, _W, _I, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
lib.gated_rmsnorm_qgemv_int4.argtypes = [_W, _P, _P, _I, _P, ctypes.c_float, _I, _P, _P, ctypes.c_size_t, _P]
lib.qgemv_q2.argtypes = [_W, _P, _I, _P, _P]
lib.moe_gather_qgemv_q2.argtypes = [_W, _W, _W, _P, _P, _I, _P, _P, _P, _P, ctypes.c_size_t, _P]
lib.moe_layer_q2.argtypes = [_P, _I, _W, _W, _W, _I, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
lib.qgemv_q2_multi.argtypes = [_I, _W, _P, _I, ctypes.POINTER(_P), _I, _P]
lib.rmsnorm_qgemv_int4.argtypes = [_W, _P, _I, _P, ctypes.c_float, _P, _P]
lib.rmsnorm_qgemv_int4_multi.argtypes = [_I, _W, _P, _I, _P, ctypes.c_float, ctypes.POINTER(_P), _I, _P]
lib.qgemv_int4_sigmoid_fma.argtypes = [_W, _P, _I, _P, _P, _P, _P, _P]
lib.sigmoid_scalar_fma_residual.argtypes = [_P, _P, _P, _P, _P, _I, _P]
lib.dense_layer_int4.argtypes = [_W, _W, _W, _P, _I, _P, _P, ctypes.c_size_t, _P]
lib.dense_layer_int4_host.argtypes = [_W, _W, _W, _P, _I, _P, _P, ctypes.c_size_t, _P]
lib.moe_gather_qgemv_int4_noalloc.argtypes = [_W, _W, _W, _P, _P, _I, _P, _P, _P, _P]
lib.scalar_fma_chain8_residual.argtypes = [_P, _P, _P, _P, _I, _P]
lib.qgemm_int4.argtypes = [_W, _P, _I, _P, _P, ctypes.c_size_t, _P]
lib.quantize_affine_q64a.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P]
lib.qgemm_int4_multi.argtypes = [_I, _W, _P, _I, ctypes.POINTER(_P), _P, ctypes.c_size_t, _P]
lib.qg_workspace_bytes.argtypes = [_I, _W, _I]
lib.qg_workspace_bytes.restype = ctypes.c_size_t
lib.qg_set_pdl.argtypes = [_I]
lib.qg_tune_gemv.argtypes = [_I]
lib.qg_tune_gemv_split.argtypes = [_I]
lib.qg_tune_qgemm.argtypes = [_I]
lib.qg_selftest_wait_timeout.argtypes = [_I, _P]
lib.qg_device_status.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32)]
lib.qg_strerror.argtypes = [_I]
lib.qg_strerror.restype = ctypes.c_char_p
lib.qg_version.argtypes = []
for _f in ("qgemv_int4", "qgemv_int4_multi", "moe_router_topk", "moe_gather_qgemv_int4",
           "moe_gather_qgemv_int4_noalloc", "moe_layer_int4", "moe_prefill_int4", "gated_rmsnorm_qgemv_int4", "dense_layer_int4", "dense_layer_int4_host", "rmsnorm_qgemv_int4", "qgemv_q2", "qgemv_q2_multi", "moe_gather_qgemv_q2", "moe_layer_q2",
           "rmsnorm_qgemv_int4_multi", "qgemv_int4_sigmoid_fma", "sigmoid_scalar_fma_residual",
           "scalar_fma_chain8_residual", "qgemm_int4", "qgemm_int4_multi", "quantize_affine_q64a", "qg_set_pdl", "qg_tune_gemv", "qg_tune_gemv_split", "qg_tune_qgemm", "qg_selftest_wait_timeout", "qg_device_status", "qg_version"):
    getattr(lib, _f).restype = ctypes.c_int


class QGError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {qg_strerror(code)} ({code})")


def _check(rc: int, where: str) -> None:
    if rc != QG_OK:
        raise QGError(rc, where)


def qg_strerror(code: int) -> str:
    return lib.qg_strerror(int(code)).decode()


# ---------------------------------------------------------------- torch marshalling
def _torch():
    import torch
    return torch


def _ptr(t) -> int:
    """Address of a device tensor for the C ABI (None -> 0).  The calls read and write flat device
    arrays, so a tensor on the host or a non-contiguous view is refused here, before any launch."""
    if t is None:
        return 0
    if not t.is_cuda:
        raise QGError(QG_EINVAL, f"expected a CUDA tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise QGError(QG_EINVAL, "expected a contiguous tensor")
    return int(t.data_ptr())


def _hptr(t) -> int:
    """Address of a host tensor for the host-buffer calls (the library checks that it is
    page-locked)."""
    if t is None:
        return 0
    if t.is_cuda:
        raise QGError(QG_EINVAL, "expected a host tensor")
    if not t.is_contiguous():
        raise QGError(QG_EINVAL, "expected a contiguous tensor")
    return int(t.data_ptr())


_DT_NAMES = {"f32": ("float32",), "bf16": ("bfloat16",), "i32": ("int32",), "x": ("bfloat16", "float32")}


def _need(what: str, n: int, *ts, dt: str) -> None:
    """The kernels read and write whole vectors of a fixed element type through plain pointers: a
    tensor of another dtype, or shorter than the call needs, is refused here (QG_EINVAL) instead
    of being read or written past its end.  dt: "f32", "bf16", "i32" (uint32 indices) or "x"
    (bf16 or fp32, the type the call is told)."""
    torch = _torch()
    ok = tuple(getattr(torch, d) for d in _DT_NAMES[dt])
    for t in ts:
        if t is None:
            continue
        if t.dtype not in ok:
            raise QGError(QG_EINVAL, f"{what}: dtype {t.dtype} where the call needs {' or '.join(_DT_NAMES[dt])}")
        if t.numel() < n:
            raise QGError(QG_EINVAL, f"{what}: {t.numel()} elements where the call needs {n}")


def _stream(stream) -> int:
    if stream is None:
        return int(_torch().cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def to_device(a: np.ndarray, device="cuda"):
    """numpy -> torch CUDA tensor with the same bytes (uint32 -> int32, uint16 bf16 bits -> bfloat16)."""
    torch = _torch()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(device)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_numpy(t) -> np.ndarray:
    torch = _torch()
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.int32:
        return t.numpy().view(np.uint32)
    return t.numpy()


class Int4Weight:
    """Device tensors of one int4 affine weight (or a stack of n_mat expert weights)."""

    def __init__(self, packed, scales, biases, out: int, in_dim: int, n_mat: int = 1, group_size: int = 64,
                 bits: int = 4):
        """bits: 4 (Q4_64A, packed [n_mat][out][in/8]) or 2 (Q2_64A, packed [n_mat][out][in/16])."""
        self.packed, self.scales, self.biases = packed, scales, biases
        self.out, self.in_dim, self.n_mat, self.group_size = int(out), int(in_dim), int(n_mat), int(group_size)
        if bits not in (2, 4):
            raise QGError(QG_EINVAL, f"bits must be 2 or 4, got {bits}")
        self.bits = bits
        if self.group_size == 64 and self.in_dim % 64 == 0 and self.out > 0 and self.n_mat > 0:
            rows = self.n_mat * self.out
            _need("packed", rows * self.in_dim * bits // 32, packed, dt="i32")
            _need("scales, biases", rows * (self.in_dim // 64), scales, biases, dt="bf16")
        self._s = qg_int4_weight(_ptr(packed), _ptr(scales), _ptr(biases), self.out, self.in_dim,
                                 self.group_size, self.n_mat)

    @classmethod
    def from_numpy(cls, d: dict, device="cuda") -> "Int4Weight":
        packed = d["packed"]
        if packed.ndim == 3:
            n_mat, out, w = packed.shape
        else:
            (out, w), n_mat = packed.shape, 1
        return cls(to_device(packed, device), to_device(d["scales"], device), to_device(d["biases"], device),
                   out, w * 8, n_mat)

    def _bits(self, bits: int, where: str) -> None:
        if self.bits != bits:
            raise QGError(QG_EINVAL, f"{where}: a {self.bits}-bit weight where the call takes {bits}-bit codes")

    @property
    def struct(self) -> qg_int4_weight:
        return self._s


def _xtype(x) -> int:
    torch = _torch()
    if x.dtype == torch.bfloat16:
        return QG_X_BF16
    if x.dtype == torch.float32:
        return QG_X_F32
    raise TypeError(f"x must be bfloat16 or float32, got {x.dtype}")


# ---------------------------------------------------------------- entry points
def qgemv_int4(w: Int4Weight, x, y=None, stream=None):
    torch = _torch()
    if y is None:
        y = torch.empty(w.out, dtype=torch.float32, device=x.device)
    _need("x", w.in_dim, x, dt="x")
    _need("y", w.out, y, dt="f32")
    w._bits(4, "qgemv_int4")
    _check(lib.qgemv_int4(ctypes.byref(w.struct), _ptr(x), _xtype(x), _ptr(y), _stream(stream)), "qgemv_int4")
    return y


def qgemv_int4_multi(ws, x, ys=None, epilogue: str = "none", stream=None):
    torch = _torch()
    n = len(ws)
    epi = {"none": QG_EPI_NONE, "swiglu": QG_EPI_SWIGLU}[epilogue]
    if ys is None:
        ys = [torch.empty(w.out, dtype=torch.float32, device=x.device) for w in ws]
        if epi == QG_EPI_SWIGLU:
            ys[1] = None
    _need("x", ws[0].in_dim, x, dt="x")
    for w, y_ in zip(ws, ys):
        _need("y", w.out, y_, dt="f32")
    arr = (qg_int4_weight * n)(*[w.struct for w in ws])
    yp = (_P * n)(*[_ptr(y) for y in ys])
    for w_ in ws:
        w_._bits(4, "qgemv_int4_multi")
    _check(lib.qgemv_int4_multi(n, arr, _ptr(x), _xtype(x), yp, epi, _stream(stream)), "qgemv_int4_multi")
    return ys[0] if epi == QG_EPI_SWIGLU else ys


def qgemv_q2(w: Int4Weight, x, y=None, stream=None):
    """2-bit affine GEMV (w.packed [out][in/16])."""
    torch = _torch()
    if y is None:
        y = torch.empty(w.out, dtype=torch.float32, device=x.device)
    _need("x", w.in_dim, x, dt="x")
    _need("y", w.out, y, dt="f32")
    w._bits(2, "qgemv_q2")
    _check(lib.qgemv_q2(ctypes.byref(w.struct), _ptr(x), _xtype(x), _ptr(y), _stream(stream)), "qgemv_q2")
    return y


def qgemv_q2_multi(ws, x, ys=None, epilogue: str = "none", stream=None):
    torch = _torch()
    n = len(ws)
    epi = {"none": QG_EPI_NONE, "swiglu": QG_EPI_SWIGLU}[epilogue]
    if ys is None:
        ys = [torch.empty(w.out, dtype=torch.float32, device=x.device) for w in ws]
        if epi == QG_EPI_SWIGLU:
            ys[1] = None
    _need("x", ws[0].in_dim, x, dt="x")
    for w, y_ in zip(ws, ys):
        _need("y", w.out, y_, dt="f32")
    arr = (qg_int4_weight * n)(*[w.struct for w in ws])
    yp = (_P * n)(*[_ptr(y) for y in ys])
    for w_ in ws:
        w_._bits(2, "qgemv_q2_multi")
    _check(lib.qgemv_q2_multi(n, arr, _ptr(x), _xtype(x), yp, epi, _stream(stream)), "qgemv_q2_multi")
    return ys[0] if epi == QG_EPI_SWIGLU else ys


def rmsnorm_qgemv_int4(w: Int4Weight, x, gamma, eps: float = 1e-6, y=None, stream=None):
    """y = W (x * gamma / sqrt(mean(x^2) + eps)); gamma bf16 [in]."""
    torch = _torch()
    if y is None:
        y = torch.empty(w.out, dtype=torch.float32, device=x.device)
    _need("x", w.in_dim, x, dt="x")
    _need("gamma", w.in_dim, gamma, dt="bf16")
    _need("y", w.out, y, dt="f32")
    w._bits(4, "rmsnorm_qgemv_int4")
    _check(lib.rmsnorm_qgemv_int4(ctypes.byref(w.struct), _ptr(x), _xtype(x), _ptr(gamma), float(eps), _ptr(y),
                                  _stream(stream)), "rmsnorm_qgemv_int4")
    return y


def rmsnorm_qgemv_int4_multi(ws, x, gamma, eps: float = 1e-6, ys=None, epilogue: str = "none", stream=None):
    torch = _torch()
    n = len(ws)
    epi = {"none": QG_EPI_NONE, "swiglu": QG_EPI_SWIGLU}[epilogue]
    if ys is None:
        ys = [torch.empty(w.out, dtype=torch.float32, device=x.device) for w in ws]
        if epi == QG_EPI_SWIGLU:
            ys[1] = None
    _need("x", ws[0].in_dim, x, dt="x")
    _need("gamma", ws[0].in_dim, gamma, dt="bf16")
    for w, y_ in zip(ws, ys):
        _need("y", w.out, y_, dt="f32")
    arr = (qg_int4_weight * n)(*[w.struct for w in ws])
    yp = (_P * n)(*[_ptr(y) for y in ys])
    for w_ in ws:
        w_._bits(4, "rmsnorm_qgemv_int4_multi")
    _check(lib.rmsnorm_qgemv_int4_multi(n, arr, _ptr(x), _xtype(x), _ptr(gamma), float(eps), yp, epi,
                                        _stream(stream)), "rmsnorm_qgemv_int4_multi")
    return ys[0] if epi == QG_EPI_SWIGLU else ys


def qgemv_int4_sigmoid_fma(w: Int4Weight, x, gate, base, residual=None, y=None, stream=None):
    """y = base + sigmoid(gate[0]) * (W x) (+ residual bf16)."""
    torch = _torch()
    if y is None:
        y = torch.empty(w.out, dtype=torch.float32, device=x.device)
    _need("x", w.in_dim, x, dt="x")
    _need("gate", 1, gate, dt="f32")
    _need("base, y", w.out, base, y, dt="f32")
    _need("residual", w.out, residual, dt="bf16")
    w._bits(4, "qgemv_int4_sigmoid_fma")
    _check(lib.qgemv_int4_sigmoid_fma(ctypes.byref(w.struct), _ptr(x), _xtype(x), _ptr(gate), _ptr(base),
                                      _ptr(residual), _ptr(y), _stream(stream)), "qgemv_int4_sigmoid_fma")
    return y


def sigmoid_scalar_fma_residual(gate, value, base, residual=None, out=None, stream=None):
    """out = base + sigmoid(gate[0]) * value (+ residual bf16)."""
    torch = _torch()
    n = value.numel()
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=value.device)
    _need("gate", 1, gate, dt="f32")
    _need("value, base, out", n, value, base, out, dt="f32")
    _need("residual", n, residual, dt="bf16")
    _check(lib.sigmoid_scalar_fma_residual(_ptr(gate), _ptr(value), _ptr(base), _ptr(residual), _ptr(out), n,
                                           _stream(stream)), "sigmoid_scalar_fma_residual")
    return out


def moe_router_topk(logits, k: int = 8, renorm: bool = True, idx=None, p=None, stream=None):
    torch = _torch()
    if idx is None:
        idx = torch.empty(k, dtype=torch.int32, device=logits.device)
    if p is None:
        p = torch.empty(k, dtype=torch.float32, device=logits.device)
    _need("logits", 1, logits, dt="f32")
    _need("idx", k, idx, dt="i32")
    _need("p", k, p, dt="f32")
    _check(lib.moe_router_topk(_ptr(logits), logits.numel(), k, 1 if renorm else 0, _ptr(idx), _ptr(p),
                               _stream(stream)), "moe_router_topk")
    return idx, p


def qg_workspace_bytes(op: int, w: Int4Weight, t_or_k: int) -> int:
    return int(lib.qg_workspace_bytes(op, ctypes.byref(w.struct), t_or_k))


def moe_gather_qgemv_int4(gate: Int4Weight, up: Int4Weight, down: Int4Weight, idx, p, x, residual, y=None,
                          workspace=None, stream=None, bits: int = 4):
    torch = _torch()
    k = idx.numel()
    if y is None:
        y = torch.empty(down.out, dtype=torch.float32, device=x.device)
    need = qg_workspace_bytes(QG_OP_MOE, down, k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _need("idx", k, idx, dt="i32")
    _need("p", k, p, dt="f32")
    _need("x", gate.in_dim, x, dt="bf16")
    _need("residual", down.out, residual, dt="bf16")
    _need("y", down.out, y, dt="f32")
    for w_ in (gate, up, down):
        w_._bits(bits, "moe_gather_qgemv")
    fn = lib.moe_gather_qgemv_int4 if bits == 4 else lib.moe_gather_qgemv_q2
    _check(fn(ctypes.byref(gate.struct), ctypes.byref(up.struct), ctypes.byref(down.struct),
              _ptr(idx), _ptr(p), k, _ptr(x), _ptr(residual), _ptr(y), _ptr(workspace),
              workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_gather_qgemv_int4" if bits == 4 else "moe_gather_qgemv_q2")
    return y


def moe_layer_int4(logits, gate: Int4Weight, up: Int4Weight, down: Int4Weight, x, residual, k: int = 8,
                   renorm: bool = True, y=None, idx=None, p=None, workspace=None, stream=None, bits: int = 4):
    """Router + expert gather in one call; returns (y, idx, p)."""
    torch = _torch()
    dev = x.device
    if y is None:
        y = torch.empty(down.out, dtype=torch.float32, device=dev)
    if idx is None:
        idx = torch.empty(k, dtype=torch.int32, device=dev)
    if p is None:
        p = torch.empty(k, dtype=torch.float32, device=dev)
    need = qg_workspace_bytes(QG_OP_MOE, down, k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _need("logits", gate.n_mat, logits, dt="f32")
    _need("x", gate.in_dim, x, dt="bf16")
    _need("residual", down.out, residual, dt="bf16")
    _need("y", down.out, y, dt="f32")
    _need("idx", k, idx, dt="i32")
    _need("p", k, p, dt="f32")
    for w_ in (gate, up, down):
        w_._bits(bits, "moe_layer")
    fn = lib.moe_layer_int4 if bits == 4 else lib.moe_layer_q2
    _check(fn(_ptr(logits), 1 if renorm else 0, ctypes.byref(gate.struct), ctypes.byref(up.struct),
              ctypes.byref(down.struct), k, _ptr(x), _ptr(residual), _ptr(y), _ptr(idx), _ptr(p),
              _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_layer_int4" if bits == 4 else "moe_layer_q2")
    return y, idx, p


def gated_rmsnorm_qgemv_int4(w: Int4Weight, y, z, gamma, eps: float, head_dim: int, out=None, workspace=None,
                             stream=None):
    """out = W (silu(z) * gamma * rmsnorm per head of y); y, z bf16 or fp32 (the same type)."""
    torch = _torch()
    if out is None:
        out = torch.empty(w.out, dtype=torch.float32, device=y.device)
    if workspace is None:
        workspace = torch.empty(qg_workspace_bytes(QG_OP_GATED_NORM, w, 0), dtype=torch.uint8, device=y.device)
    _need("y, z", w.in_dim, y, z, dt="x")
    if z.dtype != y.dtype:
        raise QGError(QG_EINVAL, "y and z must have the same dtype")
    _need("gamma", w.in_dim, gamma, dt="bf16")
    _need("out", w.out, out, dt="f32")
    w._bits(4, "gated_rmsnorm_qgemv_int4")
    _check(lib.gated_rmsnorm_qgemv_int4(ctypes.byref(w.struct), _ptr(y), _ptr(z), _xtype(y), _ptr(gamma), float(eps),
                                        int(head_dim), _ptr(out), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream)),
           "gated_rmsnorm_qgemv_int4")
    return out


def moe_prefill_int4(logits, gate: Int4Weight, up: Int4Weight, down: Int4Weight, X, residual=None, k: int = 8,
                     renorm: bool = True, Y=None, idx=None, p=None, workspace=None, stream=None):
    """The MoE layer for T tokens (prefill): logits fp32 [T][E], X bf16 [T][hidden], residual bf16
    [T][hidden] or None; returns (Y fp32 [T][hidden], idx int32 [T][k], p fp32 [T][k])."""
    torch = _torch()
    dev = X.device
    T = int(logits.shape[0])
    if Y is None:
        Y = torch.empty((T, down.out), dtype=torch.float32, device=dev)
    if idx is None:
        idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    if p is None:
        p = torch.empty((T, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(qg_workspace_bytes(QG_OP_MOE_PREFILL, down, T), 16), dtype=torch.uint8, device=dev)
    _need("logits", T * gate.n_mat, logits, dt="f32")
    _need("X, residual", T * gate.in_dim, X, residual, dt="bf16")
    _need("Y", T * down.out, Y, dt="f32")
    _need("idx", T * k, idx, dt="i32")
    _need("p", T * k, p, dt="f32")
    for w_ in (gate, up, down):
        w_._bits(4, "moe_prefill_int4")
    _check(lib.moe_prefill_int4(_ptr(logits), T, 1 if renorm else 0, ctypes.byref(gate.struct), ctypes.byref(up.struct),
                                ctypes.byref(down.struct), k, _ptr(X), _ptr(residual), _ptr(Y), _ptr(idx), _ptr(p),
                                _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_prefill_int4")
    return Y, idx, p


def dense_layer_int4(gate: Int4Weight, up: Int4Weight, down: Int4Weight, x, y=None, workspace=None, stream=None):
    """y = W_down (silu(W_g x) * (W_u x)); x bf16 or fp32.  Returns y; h (fp32 [inter]) is the
    first inter floats of the workspace after the call."""
    torch = _torch()
    dev = x.device
    if y is None:
        y = torch.empty(down.out, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(qg_workspace_bytes(QG_OP_LAYER, down, 0), dtype=torch.uint8, device=dev)
    _need("x", gate.in_dim, x, dt="x")
    _need("y", down.out, y, dt="f32")
    for w_ in (gate, up, down):
        w_._bits(4, "dense_layer_int4")
    _check(lib.dense_layer_int4(ctypes.byref(gate.struct), ctypes.byref(up.struct), ctypes.byref(down.struct),
                                _ptr(x), _xtype(x), _ptr(y), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
           "dense_layer_int4")
    return y


def dense_layer_int4_host(gate: Int4Weight, up: Int4Weight, down: Int4Weight, x_host, y_host, workspace=None,
                          stream=None, device="cuda"):
    """dense_layer_int4 with x_host (bf16 or fp32) and y_host (fp32) pinned CPU tensors; y_host is
    written by the GPU (synchronise the stream before reading it).  Returns y_host."""
    torch = _torch()
    if workspace is None:
        workspace = torch.empty(qg_workspace_bytes(QG_OP_LAYER_HOST, down, gate.in_dim), dtype=torch.uint8,
                                device=device)
    _need("x_host", gate.in_dim, x_host, dt="x")
    _need("y_host", down.out, y_host, dt="f32")
    for w_ in (gate, up, down):
        w_._bits(4, "dense_layer_int4_host")
    _check(lib.dense_layer_int4_host(ctypes.byref(gate.struct), ctypes.byref(up.struct), ctypes.byref(down.struct),
                                     _hptr(x_host), _xtype(x_host), _hptr(y_host), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)),
           "dense_layer_int4_host")
    return y_host


def moe_gather_qgemv_int4_noalloc(gate: Int4Weight, up: Int4Weight, down: Int4Weight, idx, p, x, residual, y,
                                  stream=None):
    """moe_gather_qgemv_int4 with the library's fixed scratch; `y` must be supplied (nothing is
    allocated on this path)."""
    _need("idx", idx.numel(), idx, dt="i32")
    _need("p", idx.numel(), p, dt="f32")
    _need("x", gate.in_dim, x, dt="bf16")
    _need("residual", down.out, residual, dt="bf16")
    _need("y", down.out, y, dt="f32")
    for w_ in (gate, up, down):
        w_._bits(4, "moe_gather_qgemv_int4_noalloc")
    _check(lib.moe_gather_qgemv_int4_noalloc(ctypes.byref(gate.struct), ctypes.byref(up.struct),
                                             ctypes.byref(down.struct), _ptr(idx), _ptr(p), idx.numel(), _ptr(x),
                                             _ptr(residual), _ptr(y), _stream(stream)),
           "moe_gather_qgemv_int4_noalloc")
    return y


def scalar_fma_chain8_residual(p, v, residual, out=None, stream=None):
    torch = _torch()
    n = residual.numel()
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=v.device)
    _need("p", 8, p, dt="f32")
    _need("v", 8 * n, v, dt="f32")
    _need("residual", n, residual, dt="bf16")
    _need("out", n, out, dt="f32")
    _check(lib.scalar_fma_chain8_residual(_ptr(p), _ptr(v), _ptr(residual), _ptr(out), n, _stream(stream)),
           "scalar_fma_chain8_residual")
    return out


def quantize_affine_q64a(w, bits: int = 4, stream=None):
    """Encode w (bf16 or fp32 [out][in]) in the affine group-64 format: (packed int32
    [out][in*bits/32], scales bf16 [out][in/64], biases bf16 [out][in/64])."""
    torch = _torch()
    out, in_dim = w.shape
    packed = torch.empty((out, in_dim * bits // 32), dtype=torch.int32, device=w.device)
    scales = torch.empty((out, in_dim // 64), dtype=torch.bfloat16, device=w.device)
    biases = torch.empty((out, in_dim // 64), dtype=torch.bfloat16, device=w.device)
    _check(lib.quantize_affine_q64a(_ptr(w), _xtype(w), out, in_dim, bits, _ptr(packed), _ptr(scales), _ptr(biases),
                                    _stream(stream)), "quantize_affine_q64a")
    return packed, scales, biases


def qgemm_int4_multi(ws, X, Ys=None, workspace=None, stream=None):
    """Ys[i] = X W_i^T for n in {2,3,4} weights sharing in; X bf16 [T][in]."""
    torch = _torch()
    n, T = len(ws), X.shape[0]
    if Ys is None:
        Ys = [torch.empty((T, w.out), dtype=torch.float32, device=X.device) for w in ws]
    need = qg_workspace_bytes(QG_OP_QGEMM, ws[0], T)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _need("X", T * ws[0].in_dim, X, dt="bf16")
    for w, y_ in zip(ws, Ys):
        _need("Y", T * w.out, y_, dt="f32")
    arr = (qg_int4_weight * n)(*[w.struct for w in ws])
    yp = (_P * n)(*[_ptr(y) for y in Ys])
    for w_ in ws:
        w_._bits(4, "qgemm_int4_multi")
    _check(lib.qgemm_int4_multi(n, arr, _ptr(X), T, yp, _ptr(workspace), nbytes, _stream(stream)), "qgemm_int4_multi")
    return Ys


def qgemm_int4(w: Int4Weight, X, Y=None, workspace=None, stream=None):
    torch = _torch()
    T = X.shape[0]
    if Y is None:
        Y = torch.empty((T, w.out), dtype=torch.float32, device=X.device)
    need = qg_workspace_bytes(QG_OP_QGEMM, w, T)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _need("X", T * w.in_dim, X, dt="bf16")
    _need("Y", T * w.out, Y, dt="f32")
    w._bits(4, "qgemm_int4")
    _check(lib.qgemm_int4(ctypes.byref(w.struct), _ptr(X), T, _ptr(Y), _ptr(workspace), nbytes, _stream(stream)),
           "qgemm_int4")
    return Y


def qg_set_pdl(enable: bool) -> bool:
    return bool(lib.qg_set_pdl(1 if enable else 0))


def qg_tune_gemv(ctas_per_sm: int = 0) -> None:
    _check(lib.qg_tune_gemv(ctas_per_sm), "qg_tune_gemv")


def qg_tune_gemv_split(kcl: int = 0) -> None:
    """K split of the GEMV across a thread-block cluster: 0 automatic, 1 never, 2..4 forced."""
    _check(lib.qg_tune_gemv_split(kcl), "qg_tune_gemv_split")


def qg_selftest_wait_timeout(limit_us: int = 1000, stream=None) -> None:
    _check(lib.qg_selftest_wait_timeout(limit_us, _stream(stream)), "qg_selftest_wait_timeout")


def qg_tune_qgemm(tc_min_T: int = 0) -> None:
    _check(lib.qg_tune_qgemm(tc_min_T), "qg_tune_qgemm")


def qg_device_status(stream=None) -> int:
    s = ctypes.c_uint32(0)
    _check(lib.qg_device_status(_stream(stream), ctypes.byref(s)), "qg_device_status")
    return int(s.value)


def qg_version() -> int:
    return int(lib.qg_version())

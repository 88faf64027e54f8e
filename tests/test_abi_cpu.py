"""The C ABI library builds for sm_103a, loads, exports every entry point include/qg.h declares,
and rejects bad arguments on the host before touching a GPU.  CPU only: every call below fails
validation, so no CUDA runtime call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qg.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|void)\s*\**\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from moe_int4_affine_gb300 import build

    return ctypes.CDLL(build.build())


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ["qgemv_int4", "qgemv_int4_multi", "moe_router_topk", "moe_gather_qgemv_int4",
              "scalar_fma_chain8_residual", "qgemm_int4", "qg_workspace_bytes", "qg_device_status",
              "qg_strerror", "qg_set_pdl", "qg_version"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), f"libqg.so does not export {n}"


class W(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p),
                ("out", ctypes.c_int32), ("in_", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("n_mat", ctypes.c_int32)]


FAKE = 0x10000  # an aligned non-null address; never dereferenced (validation fails first)


def _w(**kw):
    d = dict(packed=FAKE, scales=FAKE, biases=FAKE, out=8, in_=128, group_size=64, n_mat=1)
    d.update(kw)
    return W(**d)


def test_host_validation_error_codes(lib):
    P = ctypes.c_void_p
    lib.qgemv_int4.argtypes = [ctypes.POINTER(W), P, ctypes.c_int, P, P]
    call = lambda w, x=FAKE, xt=0, y=FAKE: lib.qgemv_int4(ctypes.byref(w), x, xt, y, None)
    assert call(_w(group_size=32)) == -1
    assert call(_w(in_=96)) == -1
    assert call(_w(in_=0)) == -1
    assert call(_w(out=0)) == -1
    assert call(_w(n_mat=2)) == -1
    assert call(_w(packed=None)) == -1
    assert call(_w(), x=None) == -1
    assert call(_w(), xt=7) == -1
    assert call(_w(in_=65536)) == -5
    assert call(_w(scales=FAKE + 2)) == -2
    assert call(_w(), x=FAKE + 8) == -2
    assert call(_w(), y=FAKE + 4) == -2
    lib.qgemv_int4_multi.argtypes = [ctypes.c_int, ctypes.POINTER(W), P, ctypes.c_int, ctypes.POINTER(P),
                                     ctypes.c_int, P]
    ws = (W * 2)(_w(), _w(in_=256))
    ys = (P * 2)(FAKE, FAKE)
    assert lib.qgemv_int4_multi(2, ws, FAKE, 0, ys, 0, None) == -1  # mismatched widths
    ws = (W * 2)(_w(), _w(out=9))
    assert lib.qgemv_int4_multi(2, ws, FAKE, 0, ys, 1, None) == -1  # swiglu needs equal outs
    assert lib.qgemv_int4_multi(5, ws, FAKE, 0, ys, 0, None) == -1
    lib.moe_router_topk.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P]
    assert lib.moe_router_topk(FAKE, 4, 5, 1, FAKE, FAKE, None) == -1
    assert lib.moe_router_topk(FAKE, 2048, 8, 1, FAKE, FAKE, None) == -5
    assert lib.moe_router_topk(FAKE, 128, 8, 2, FAKE, FAKE, None) == -1
    lib.moe_gather_qgemv_int4.argtypes = [ctypes.POINTER(W)] * 3 + [P, P, ctypes.c_int, P, P, P, P,
                                                                     ctypes.c_size_t, P]
    g, u, dn = _w(out=64, in_=128, n_mat=4), _w(out=64, in_=128, n_mat=4), _w(out=128, in_=64, n_mat=4)
    args = lambda k=8, ws=FAKE, nb=1 << 20, d=dn: (ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), FAKE, FAKE, k,
                                                   FAKE, FAKE, FAKE, ws, nb, None)
    assert lib.moe_gather_qgemv_int4(*args(k=9)) == -1
    assert lib.moe_gather_qgemv_int4(*args(ws=None)) == -3
    assert lib.moe_gather_qgemv_int4(*args(nb=100)) == -3
    assert lib.moe_gather_qgemv_int4(*args(d=_w(out=128, in_=128, n_mat=4))) == -1
    lib.scalar_fma_chain8_residual.argtypes = [P, P, P, P, ctypes.c_int, P]
    assert lib.scalar_fma_chain8_residual(FAKE, FAKE, FAKE, FAKE, 0, None) == -1
    assert lib.scalar_fma_chain8_residual(FAKE, FAKE + 4, FAKE, FAKE, 8, None) == -2
    lib.qgemm_int4.argtypes = [ctypes.POINTER(W), P, ctypes.c_int, P, P, ctypes.c_size_t, P]
    assert lib.qgemm_int4(ctypes.byref(_w()), FAKE, 0, FAKE, None, 0, None) == -1
    assert lib.qgemm_int4(ctypes.byref(_w()), FAKE, 5000, FAKE, None, 0, None) == -1


def test_workspace_and_strings(lib):
    lib.qg_workspace_bytes.argtypes = [ctypes.c_int, ctypes.POINTER(W), ctypes.c_int]
    lib.qg_workspace_bytes.restype = ctypes.c_size_t
    down = _w(out=2048, in_=768, n_mat=128)
    assert lib.qg_workspace_bytes(2, ctypes.byref(down), 8) == 8 * 768 * 4
    assert lib.qg_workspace_bytes(0, ctypes.byref(down), 8) == 0
    lib.qg_strerror.restype = ctypes.c_char_p
    assert lib.qg_strerror(-3) == b"workspace missing or too small"
    assert lib.qg_set_pdl(1) == 0 and lib.qg_set_pdl(0) == 1
    assert lib.qg_version() >> 16 == 1


def test_host_validation_of_the_later_entry_points(lib):
    """moe_prefill_int4, gated_rmsnorm_qgemv_int4 and quantize_affine_q64a reject bad arguments on
    the host (every call here fails validation)."""
    P = ctypes.c_void_p
    lib.moe_prefill_int4.argtypes = [P, ctypes.c_int, ctypes.c_int] + [ctypes.POINTER(W)] * 3 + \
        [ctypes.c_int, P, P, P, P, P, P, ctypes.c_size_t, P]
    g, u, dn = _w(out=64, in_=128, n_mat=8), _w(out=64, in_=128, n_mat=8), _w(out=128, in_=64, n_mat=8)
    pre = lambda T=4, k=2, ws=FAKE, nb=1 << 30, d=dn, renorm=1, res=FAKE: lib.moe_prefill_int4(
        FAKE, T, renorm, ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), k, FAKE, res, FAKE, FAKE, FAKE, ws, nb, None)
    assert pre(k=9) == -1
    assert pre(k=0) == -1
    assert pre(T=0) == -1
    assert pre(T=70000) == -1
    assert pre(renorm=2) == -1
    assert pre(d=_w(out=128, in_=128, n_mat=8)) == -1  # down's in must be the intermediate size
    assert pre(ws=None) == -3
    assert pre(nb=1000) == -3
    assert pre(res=FAKE + 8) == -2
    lib.gated_rmsnorm_qgemv_int4.argtypes = [ctypes.POINTER(W), P, P, ctypes.c_int, P, ctypes.c_float, ctypes.c_int,
                                             P, P, ctypes.c_size_t, P]
    w = _w(out=8, in_=256)
    gated = lambda hd=128, z=FAKE, eps=1e-6, ws=FAKE, nb=4096, xt=0: lib.gated_rmsnorm_qgemv_int4(
        ctypes.byref(w), FAKE, z, xt, FAKE, eps, hd, FAKE, ws, nb, None)
    assert gated(hd=0) == -1
    assert gated(hd=96) == -1  # does not divide in
    assert gated(hd=512) == -1
    assert gated(z=None) == -1
    assert gated(eps=-1.0) == -1
    assert gated(xt=3) == -1
    assert gated(nb=100) == -3
    assert gated(z=FAKE + 4) == -2
    lib.quantize_affine_q64a.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P]
    q = lambda bits=4, out=8, in_=128, wt=0, w_=FAKE: lib.quantize_affine_q64a(w_, wt, out, in_, bits, FAKE, FAKE,
                                                                              FAKE, None)
    assert q(bits=3) == -1
    assert q(in_=100) == -1
    assert q(out=0) == -1
    assert q(wt=5) == -1
    assert q(w_=FAKE + 2) == -2


def test_workspace_sizes_of_the_later_ops(lib):
    lib.qg_workspace_bytes.argtypes = [ctypes.c_int, ctypes.POINTER(W), ctypes.c_int]
    lib.qg_workspace_bytes.restype = ctypes.c_size_t
    w = _w(out=2048, in_=4096)
    assert lib.qg_workspace_bytes(7, ctypes.byref(w), 0) == 4096 * 4  # gated norm: x fp32 [in]
    down = _w(out=2048, in_=768, n_mat=128)
    sizes = [lib.qg_workspace_bytes(6, ctypes.byref(down), T) for T in (1, 32, 256, 512)]
    # at least the grouped rows' token tiles, gate/up outputs, h tiles and down outputs for T k rows
    for T, b in zip((1, 32, 256, 512), sizes):
        rows = T * 8
        assert b >= rows * (2048 * 2 + 768 * 4 * 2 + 768 * 2 + 2048 * 4)
    assert sizes == sorted(sizes)
    assert lib.qg_workspace_bytes(6, ctypes.byref(down), 0) == 0


def test_binding_refuses_host_and_strided_tensors():
    """The Python binding passes flat device arrays to the C ABI: a host tensor or a strided view
    where device memory is expected is refused before any call (QG_EINVAL)."""
    torch = pytest.importorskip("torch")
    from moe_int4_affine_gb300 import qg

    with pytest.raises(qg.QGError) as e:
        qg._ptr(torch.zeros(8))
    assert e.value.code == qg.QG_EINVAL
    t = torch.zeros(4, 4)
    with pytest.raises(qg.QGError):
        qg._hptr(t.t())  # a transposed (non-contiguous) view
    assert qg._hptr(t) == t.data_ptr()
    assert qg._ptr(None) == 0 and qg._hptr(None) == 0


def test_binding_refuses_short_vectors():
    """A vector shorter than the call needs is refused before the call (QG_EINVAL), not read or
    written past its end by a kernel."""
    torch = pytest.importorskip("torch")
    from moe_int4_affine_gb300 import qg

    qg._need("x", 4, torch.zeros(4), None, dt="f32")
    with pytest.raises(qg.QGError) as e:
        qg._need("x", 5, torch.zeros(4), dt="f32")
    assert e.value.code == qg.QG_EINVAL and "x" in str(e.value)


@pytest.mark.parametrize("dt,bad", [("f32", "bfloat16"), ("f32", "float16"), ("i32", "int8"), ("i32", "int16"),
                                    ("i32", "int64"), ("bf16", "float16"), ("bf16", "float32"), ("x", "float16"),
                                    ("x", "int32")])
def test_binding_refuses_wrong_dtypes(dt, bad):
    """A tensor of the right length but another element type (a bf16 y where the kernel writes
    4-byte floats, an int8 idx where it reads 4-byte indices) is refused before the call: its
    bytes would not cover what the kernel reads or writes."""
    torch = pytest.importorskip("torch")
    from moe_int4_affine_gb300 import qg

    t = torch.zeros(64, dtype=getattr(torch, bad))
    with pytest.raises(qg.QGError) as e:
        qg._need("arg", 64, t, dt=dt)
    assert e.value.code == qg.QG_EINVAL and "dtype" in str(e.value)
    good = {"f32": torch.float32, "i32": torch.int32, "bf16": torch.bfloat16, "x": torch.bfloat16}[dt]
    qg._need("arg", 64, torch.zeros(64, dtype=good), dt=dt)


def test_binding_weight_checks_sizes_and_types():
    """An Int4Weight whose packed codes are not int32, whose scales are not bf16, or whose arrays
    are shorter than out x in (x n_mat) needs for its code width, is refused when it is made."""
    torch = pytest.importorskip("torch")
    from moe_int4_affine_gb300 import qg

    def w(packed_n, sb_n, pdt=torch.int32, sdt=torch.bfloat16, bits=4, n_mat=1):
        return qg.Int4Weight(torch.zeros(packed_n, dtype=pdt), torch.zeros(sb_n, dtype=sdt),
                             torch.zeros(sb_n, dtype=sdt), 4, 128, n_mat=n_mat, bits=bits)

    # (the binding refuses host tensors only when it takes their device address: pass checks first)
    for bad in (dict(packed_n=63, sb_n=8), dict(packed_n=64, sb_n=7), dict(packed_n=64, sb_n=8, pdt=torch.float32),
                dict(packed_n=64, sb_n=8, sdt=torch.float16), dict(packed_n=31, sb_n=8, bits=2),
                dict(packed_n=64, sb_n=8, n_mat=2)):
        with pytest.raises(qg.QGError) as e:
            w(**bad)
        assert e.value.code == qg.QG_EINVAL
        assert "dtype" in str(e.value) or "elements" in str(e.value), str(e.value)
    with pytest.raises(qg.QGError) as e:
        w(packed_n=64, sb_n=8, bits=3)
    assert "bits" in str(e.value)
    # a well-formed weight gets past these checks (and is then refused only for being on the host)
    with pytest.raises(qg.QGError) as e:
        w(packed_n=64, sb_n=8)
    assert "CUDA tensor" in str(e.value)

"""GPU parity of the steps either side of the decode GEMV: the RMSNorm-fused GEMV prologue
(rmsnorm_qgemv_int4, rmsnorm_qgemv_int4_multi) and the shared-expert sigmoid-gated FMA with the
residual (qgemv_int4_sigmoid_fma, fused into the GEMV's finisher; sigmoid_scalar_fma_residual on
its own), each against the fp64 oracle through the C ABI, within |y - y_ref| <= 1e-3 * absref + 1e-6."""
import math

import numpy as np
import pytest

import oracle
from conftest import ABS, REL, assert_within, assert_within_bound, swiglu_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _x(kind, seed, n):
    return I.bf16_normal(seed, I.TID_X, n) if kind == "bf16" else I.f32_normal(seed, I.TID_X, n)


# x of 80 groups is staged by one bulk copy, of 129 groups loaded by the threads: both paths
@pytest.mark.parametrize("out,in_dim", [(256, 1024), (1000, 5120), (700, 8256), (96, 64)])
@pytest.mark.parametrize("kind", ["bf16", "f32"])
@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_rmsnorm_qgemv_vs_oracle(qg, out, in_dim, kind, eps):
    d = I.int4_weight(out + in_dim, I.TID_W, out, in_dim)
    x = _x(kind, in_dim, in_dim)
    gamma = I.bf16_normal(in_dim + 1, I.TID_RESID, in_dim)
    y = qg.rmsnorm_qgemv_int4(qg.Int4Weight.from_numpy(d), qg.to_device(x), qg.to_device(gamma), eps)
    y_ref, a = oracle.rmsnorm_qgemv(d["packed"], d["scales"], d["biases"], x, gamma, eps)
    assert_within_bound(qg.to_numpy(y).astype(np.float64), y_ref, a)
    assert qg.qg_device_status() == 0


def test_rmsnorm_qgemv_full_size_sampled(qg):
    """The norm-fused projection at the decode layer's width (17408 x 5120), rows sampled."""
    d = I.int4_weight(0, I.TID_GATE, 17408, 5120)
    x = I.bf16_normal(0, I.TID_X, 5120)
    gamma = I.bf16_normal(1, I.TID_RESID, 5120)
    y = qg.to_numpy(qg.rmsnorm_qgemv_int4(qg.Int4Weight.from_numpy(d), qg.to_device(x), qg.to_device(gamma),
                                          1e-6)).astype(np.float64)
    xn = oracle.rmsnorm(x, gamma, 1e-6)
    rng = np.random.default_rng(5)
    rows = sorted(set([0, 17407, 114, 115] + list(rng.integers(0, 17408, 60))))
    for r in rows:
        d1 = {k: d[k].reshape(17408, -1)[r:r + 1] for k in ("packed", "scales", "biases")}
        yr, ar = oracle.qgemv_f64x(d1["packed"], d1["scales"], d1["biases"], xn)
        assert_within_bound(y[r:r + 1], yr, ar, what=f"row {r}")


def test_rmsnorm_qgemv_one_hot_and_scale_invariance(qg):
    """One-hot x (eps 0): y = sqrt(n) sign(a) gamma_j W[:, j]; and y(8 x) = y(x) with eps 0."""
    out, n, j = 300, 2048, 1500
    d = I.int4_weight(2, I.TID_W, out, n)
    w = qg.Int4Weight.from_numpy(d)
    gamma = I.bf16_normal(2, I.TID_RESID, n)
    gd = qg.to_device(gamma)
    x = np.zeros(n, np.float32)
    x[j] = -3.0
    y = qg.to_numpy(qg.rmsnorm_qgemv_int4(w, qg.to_device(x), gd, 0.0)).astype(np.float64)
    y_ref, a = oracle.rmsnorm_qgemv(d["packed"], d["scales"], d["biases"], x, gamma, 0.0)
    assert_within_bound(y, y_ref, a)
    xb = I.bf16_normal(3, I.TID_X, n)
    xs = (oracle_vals(xb) * 8.0).astype(np.float32)
    y1 = qg.to_numpy(qg.rmsnorm_qgemv_int4(w, qg.to_device(xb), gd, 0.0)).astype(np.float64)
    y8 = qg.to_numpy(qg.rmsnorm_qgemv_int4(w, qg.to_device(xs), gd, 0.0)).astype(np.float64)
    y_ref, a = oracle.rmsnorm_qgemv(d["packed"], d["scales"], d["biases"], xb, gamma, 0.0)
    assert_within_bound(y1, y_ref, a)
    assert_within_bound(y8, y_ref, a, what="8x")


def oracle_vals(bits):
    return np.array([oracle.bf16_to_f64(int(b)) for b in bits])


@pytest.mark.parametrize("out,in_dim", [(17408, 5120), (500, 576)])
def test_rmsnorm_swiglu_pair(qg, out, in_dim):
    """Post-norm FFN input: h = silu(W_g xn) * (W_u xn), xn = rmsnorm(x)."""
    gd = I.int4_weight(1, I.TID_GATE, out, in_dim)
    ud = I.int4_weight(1, I.TID_UP, out, in_dim)
    x = I.bf16_normal(1, I.TID_X, in_dim)
    gamma = I.bf16_normal(2, I.TID_RESID, in_dim)
    h = qg.rmsnorm_qgemv_int4_multi([qg.Int4Weight.from_numpy(gd), qg.Int4Weight.from_numpy(ud)], qg.to_device(x),
                                    qg.to_device(gamma), 1e-6, epilogue="swiglu")
    h = qg.to_numpy(h).astype(np.float64)
    xn = oracle.rmsnorm(x, gamma, 1e-6)
    g, ag = oracle.qgemv_f64x(gd["packed"], gd["scales"], gd["biases"], xn)
    u, au = oracle.qgemv_f64x(ud["packed"], ud["scales"], ud["biases"], xn)
    # every row, within the GEMV bounds on g and u carried through SwiGLU
    assert_within(h, oracle.swiglu(g, u), swiglu_bound(g, u, REL * ag + ABS, REL * au + ABS))
    assert qg.qg_device_status() == 0


def test_rmsnorm_multi_quartet(qg):
    """A norm before a shared-input projection set (qkv/z/b/a quartet, in 2048)."""
    outs = (8192, 4096, 32, 32)
    ds = [I.int4_weight(4, I.TID_MULTI + i, o, 2048) for i, o in enumerate(outs)]
    x = I.bf16_normal(4, I.TID_X, 2048)
    gamma = I.bf16_normal(5, I.TID_RESID, 2048)
    ys = qg.rmsnorm_qgemv_int4_multi([qg.Int4Weight.from_numpy(d) for d in ds], qg.to_device(x), qg.to_device(gamma),
                                     1e-6)
    for d, y in zip(ds, ys):
        y_ref, a = oracle.rmsnorm_qgemv(d["packed"], d["scales"], d["biases"], x, gamma, 1e-6)
        assert_within_bound(qg.to_numpy(y).astype(np.float64), y_ref, a)


def _shared_ref(d, x, gate, base, resid):
    v, av = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    s = 1.0 / (1.0 + math.exp(-float(gate)))
    r = oracle_vals(resid) if resid is not None else 0.0
    return base.astype(np.float64) + s * v + r, np.abs(base.astype(np.float64)) + s * av + np.abs(r)


@pytest.mark.parametrize("out,in_dim", [(2048, 512), (5120, 17408), (37, 1024)])
@pytest.mark.parametrize("with_resid", [True, False])
def test_qgemv_sigmoid_fma_vs_oracle(qg, out, in_dim, with_resid):
    """Shared-expert down projection with the sigmoid gate, the routed output as base and the
    residual folded in: y = base + sigmoid(g) (W h) + r."""
    d = I.int4_weight(6, I.TID_DOWN, out, in_dim)
    x = I.f32_normal(6, I.TID_X, in_dim)
    gate = np.array([0.37], np.float32)
    base = I.f32_normal(7, I.TID_RESID, out)
    resid = I.bf16_normal(8, I.TID_RESID, out) if with_resid else None
    y = qg.qgemv_int4_sigmoid_fma(qg.Int4Weight.from_numpy(d), qg.to_device(x), qg.to_device(gate),
                                  qg.to_device(base), None if resid is None else qg.to_device(resid))
    y_ref, a = _shared_ref(d, x, gate[0], base, resid)
    assert_within_bound(qg.to_numpy(y).astype(np.float64), y_ref, a)
    assert qg.qg_device_status() == 0


def test_qgemv_sigmoid_fma_in_place_and_saturated_gates(qg):
    """y may overwrite base; a gate of -40 leaves base + r, +40 adds the full GEMV."""
    out, in_dim = 1024, 2048
    d = I.int4_weight(9, I.TID_DOWN, out, in_dim)
    w = qg.Int4Weight.from_numpy(d)
    x = I.bf16_normal(9, I.TID_X, in_dim)
    base = I.f32_normal(10, I.TID_RESID, out)
    resid = I.bf16_normal(11, I.TID_RESID, out)
    for g in (-40.0, 40.0, 0.0):
        bd = qg.to_device(base)
        qg.qgemv_int4_sigmoid_fma(w, qg.to_device(x), qg.to_device(np.array([g], np.float32)), bd,
                                  qg.to_device(resid), y=bd)
        y_ref, a = _shared_ref(d, x, g, base, resid)
        assert_within_bound(qg.to_numpy(bd).astype(np.float64), y_ref, a, what=f"gate {g}")


@pytest.mark.parametrize("n", [2048, 2047, 1, 5120])
@pytest.mark.parametrize("with_resid", [True, False])
def test_sigmoid_scalar_fma_residual(qg, n, with_resid):
    v = I.f32_normal(12, I.TID_X, n)
    base = I.f32_normal(13, I.TID_RESID, n)
    resid = I.bf16_normal(14, I.TID_RESID, n) if with_resid else None
    gate = np.array([-0.8], np.float32)
    out = qg.sigmoid_scalar_fma_residual(qg.to_device(gate), qg.to_device(v), qg.to_device(base),
                                         None if resid is None else qg.to_device(resid))
    y_ref, a = oracle.sigmoid_scalar_fma(float(gate[0]), v, base, resid)
    assert_within_bound(qg.to_numpy(out).astype(np.float64), y_ref, a)
    assert qg.qg_device_status() == 0


# ---------------------------------------------------------------- gated RMSNorm before a projection
@pytest.mark.parametrize("out,in_dim,head_dim", [(2048, 4096, 128), (256, 1024, 64), (500, 576, 576), (96, 512, 512),
                                                  (300, 576, 96), (128, 1024, 32), (64, 8256, 192)])
@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_gated_rmsnorm_qgemv_vs_oracle(qg, out, in_dim, head_dim, kind):
    """W (silu(z) * gamma * rmsnorm per head of y): the GDN tail shape (32 heads of 128 into 2048),
    whole-vector norms (both in the GEMV's prologue; x of 129 groups is loaded by the threads, not
    staged) and heads of 96 and 32 columns (the separate norm kernel); y and z of either type."""
    d = I.int4_weight(out + head_dim, I.TID_W, out, in_dim)
    y = _x(kind, in_dim + 1, in_dim)
    z = _x(kind, in_dim + 2, in_dim)
    gamma = I.bf16_normal(in_dim + 3, I.TID_RESID, in_dim)
    o = qg.gated_rmsnorm_qgemv_int4(qg.Int4Weight.from_numpy(d), qg.to_device(y), qg.to_device(z),
                                    qg.to_device(gamma), 1e-6, head_dim)
    y_ref, a = oracle.gated_rmsnorm_qgemv(d["packed"], d["scales"], d["biases"], y, z, gamma, 1e-6, head_dim)
    assert_within_bound(qg.to_numpy(o).astype(np.float64), y_ref, a)
    assert qg.qg_device_status() == 0


def test_gated_rmsnorm_qgemv_rejects_bad_heads_and_workspace(qg):
    import torch

    d = I.int4_weight(1, I.TID_W, 64, 256)
    w = qg.Int4Weight.from_numpy(d)
    y = qg.to_device(I.bf16_normal(1, I.TID_X, 256))
    g = qg.to_device(I.bf16_normal(2, I.TID_RESID, 256))
    for hd in (0, 96, 512):
        with pytest.raises(qg.QGError) as e:
            qg.gated_rmsnorm_qgemv_int4(w, y, y, g, 1e-6, hd)
        assert e.value.code == qg.QG_EINVAL
    with pytest.raises(qg.QGError) as e:
        qg.gated_rmsnorm_qgemv_int4(w, y, y, g, 1e-6, 128, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == qg.QG_EWORKSPACE
    assert qg.qg_device_status() == 0

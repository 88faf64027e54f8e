"""GPU parity of the 2-bit affine variant (Q2_64A: sixteen 2-bit codes per u32) of the GEMV and
the shared-input multi GEMV against the oracle's 2-bit GEMV, within
|y - y_ref| <= 1e-3 * absref + 1e-6; and the 2-bit encoder's output fed to it."""
import numpy as np
import pytest

import oracle
from conftest import ORACLE_THREADS, assert_within_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _w(qg, d, out, in_dim):
    t = qg.to_device
    return qg.Int4Weight(t(d["packed"]), t(d["scales"]), t(d["biases"]), out, in_dim, bits=2)


@pytest.mark.parametrize("out,in_dim", [(3, 64), (256, 1024), (1000, 576), (700, 8256), (130, 2048)])
@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_qgemv_q2_vs_oracle(qg, out, in_dim, kind):
    d = I.int2_weight(out, I.TID_W, out, in_dim)
    x = I.bf16_normal(in_dim, I.TID_X, in_dim) if kind == "bf16" else I.f32_normal(in_dim, I.TID_X, in_dim)
    y = qg.to_numpy(qg.qgemv_q2(_w(qg, d, out, in_dim), qg.to_device(x))).astype(np.float64)
    y_ref, a = oracle.qgemv2(d["packed"], d["scales"], d["biases"], x)
    assert_within_bound(y, y_ref, a)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("out,in_dim", [(17408, 5120), (5120, 17408)])
def test_qgemv_q2_full_size_every_row(qg, out, in_dim):
    d = I.int2_weight(0, I.TID_W, out, in_dim)
    x = I.bf16_normal(0, I.TID_X, in_dim)
    y = qg.to_numpy(qg.qgemv_q2(_w(qg, d, out, in_dim), qg.to_device(x))).astype(np.float64)
    y_ref, a = oracle.qgemv2(d["packed"], d["scales"], d["biases"], x, threads=ORACLE_THREADS)
    assert_within_bound(y, y_ref, a)


def test_qgemv_q2_multi_and_swiglu(qg):
    outs = (8192, 4096, 32, 32)
    ds = [I.int2_weight(1, I.TID_MULTI + i, o, 2048) for i, o in enumerate(outs)]
    x = I.bf16_normal(1, I.TID_X, 2048)
    ys = qg.qgemv_q2_multi([_w(qg, d, o, 2048) for d, o in zip(ds, outs)], qg.to_device(x))
    for d, y in zip(ds, ys):
        y_ref, a = oracle.qgemv2(d["packed"], d["scales"], d["biases"], x)
        assert_within_bound(qg.to_numpy(y).astype(np.float64), y_ref, a)
    g = I.int2_weight(2, I.TID_GATE, 1000, 2048)
    u = I.int2_weight(2, I.TID_UP, 1000, 2048)
    h = qg.to_numpy(qg.qgemv_q2_multi([_w(qg, g, 1000, 2048), _w(qg, u, 1000, 2048)], qg.to_device(x),
                                      epilogue="swiglu")).astype(np.float64)
    gr, ag = oracle.qgemv2(g["packed"], g["scales"], g["biases"], x)
    ur, au = oracle.qgemv2(u["packed"], u["scales"], u["biases"], x)
    h_ref = oracle.swiglu(gr, ur)
    s = 1.0 / (1.0 + np.exp(-gr))
    bound = np.abs(s * (1.0 + gr * (1.0 - s)) * ur) * ag + np.abs(gr * s) * au + np.abs(h_ref) * 1e-3
    assert_within_bound(h, h_ref, bound)
    assert qg.qg_device_status() == 0


def test_q2_encoder_feeds_the_q2_gemv(qg):
    rng = np.random.default_rng(5)
    w = rng.normal(0, 0.02, (640, 1024)).astype(np.float32)
    p, s, b = qg.quantize_affine_q64a(qg.to_device(w), 2)
    W = qg.Int4Weight(p, s, b, 640, 1024, bits=2)
    x = I.bf16_normal(5, I.TID_X, 1024)
    y = qg.to_numpy(qg.qgemv_q2(W, qg.to_device(x))).astype(np.float64)
    pr, sr, br = oracle.quantize(w, 2)
    y_ref, a = oracle.qgemv2(pr, sr, br, x)
    assert_within_bound(y, y_ref, a)


def _stack(qg, d, E, out, in_dim):
    t = qg.to_device
    return qg.Int4Weight(t(d["packed"]), t(d["scales"]), t(d["biases"]), out, in_dim, n_mat=E, bits=2)


@pytest.mark.parametrize("E,hidden,inter,k", [(128, 2048, 768, 8), (9, 576, 128, 8), (5, 256, 192, 3)])
def test_moe_q2_vs_oracle(qg, E, hidden, inter, k):
    """The 2-bit MoE step: expert gather with the device router's selection, and the layer call
    with the router inside the gate/up kernel; both against the oracle's 2-bit MoE."""
    g = I.int2_weight(E, I.TID_GATE, inter, hidden, n_mat=E)
    u = I.int2_weight(E, I.TID_UP, inter, hidden, n_mat=E)
    d = I.int2_weight(E, I.TID_DOWN, hidden, inter, n_mat=E)
    G, U, D = _stack(qg, g, E, inter, hidden), _stack(qg, u, E, inter, hidden), _stack(qg, d, E, hidden, inter)
    logits = I.f32_normal(E, I.TID_LOGITS, E)
    x = I.bf16_normal(E, I.TID_X, hidden)
    r = I.bf16_normal(E, I.TID_RESID, hidden)
    lg, xd, rd = qg.to_device(logits), qg.to_device(x), qg.to_device(r)
    i_ref, p_ref = oracle.router_topk(logits, k)
    t = lambda w: (w["packed"], w["scales"], w["biases"])
    y_ref, a, flags = oracle.moe2(t(g), t(u), t(d), i_ref, p_ref, x, r)
    assert flags == 0
    idx, p = qg.moe_router_topk(lg, k=k)
    y1 = qg.to_numpy(qg.moe_gather_qgemv_int4(G, U, D, idx, p, xd, rd, bits=2)).astype(np.float64)
    assert_within_bound(y1, y_ref, a, what="gather")
    y2, idx2, _ = qg.moe_layer_int4(lg, G, U, D, xd, rd, k=k, bits=2)
    assert qg.to_numpy(idx2).astype(np.uint32).tolist() == i_ref.tolist()
    assert_within_bound(qg.to_numpy(y2).astype(np.float64), y_ref, a, what="layer")
    assert qg.qg_device_status() == 0

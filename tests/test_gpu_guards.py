"""Out-of-bounds writes: every output, workspace and index array of a call sits between two
sentinel-filled guard regions (conftest.Guarded), and the guards are read back after the call.
The shapes are the ragged ones where an over-long write would happen (one-row outputs, row counts
off the CTA and tile multiples, token counts off the 16 / 32 / 128 tile multiples).  The values
themselves are checked elsewhere; here a kernel that writes one element too many fails even when
every value it was asked for is right."""
import numpy as np
import pytest
import torch

from conftest import Guarded
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu
f32, bf16, i32, u8 = torch.float32, torch.bfloat16, torch.int32, torch.uint8


def _intact(*bufs):
    torch.cuda.synchronize()
    for b in bufs:
        assert b.intact(), "a kernel wrote outside its buffer"


@pytest.mark.parametrize("out,in_dim", [(1, 64), (7, 64), (33, 128), (129, 17408), (5121, 576), (300, 1088)])
@pytest.mark.parametrize("xkind", ["bf16", "f32"])
def test_qgemv_guards(qg, out, in_dim, xkind):
    W = qg.Int4Weight.from_numpy(I.int4_weight(1, I.TID_W, out, in_dim))
    x = I.bf16_normal(1, I.TID_X, in_dim) if xkind == "bf16" else I.f32_normal(1, I.TID_X, in_dim)
    y = Guarded(out, f32)
    qg.qgemv_int4(W, qg.to_device(x), y=y.t)
    _intact(y)


@pytest.mark.parametrize("outs", [(3, 5), (100, 1, 37), (8192, 4096, 32, 32), (129, 257, 1, 63)])
def test_multi_guards(qg, outs):
    Ws = [qg.Int4Weight.from_numpy(I.int4_weight(2, I.TID_MULTI + i, o, 576)) for i, o in enumerate(outs)]
    ys = [Guarded(o, f32) for o in outs]
    qg.qgemv_int4_multi(Ws, qg.to_device(I.bf16_normal(2, I.TID_X, 576)), ys=[y.t for y in ys])
    _intact(*ys)


@pytest.mark.parametrize("out,in_dim", [(1, 64), (33, 1088), (17409, 256)])
def test_pair_and_norm_guards(qg, out, in_dim):
    G = qg.Int4Weight.from_numpy(I.int4_weight(3, I.TID_GATE, out, in_dim))
    U = qg.Int4Weight.from_numpy(I.int4_weight(3, I.TID_UP, out, in_dim))
    x = qg.to_device(I.bf16_normal(3, I.TID_X, in_dim))
    h = Guarded(out, f32)
    qg.qgemv_int4_multi([G, U], x, ys=[h.t, None], epilogue="swiglu")
    gamma = qg.to_device(I.bf16_normal(4, I.TID_RESID, in_dim))
    h2 = Guarded(out, f32)
    qg.rmsnorm_qgemv_int4_multi([G, U], x, gamma, 1e-6, ys=[h2.t, None], epilogue="swiglu")
    y3 = Guarded(out, f32)
    qg.rmsnorm_qgemv_int4(G, x, gamma, 1e-6, y=y3.t)
    _intact(h, h2, y3)


@pytest.mark.parametrize("head_dim", [64, 96, 128])
def test_gated_norm_guards(qg, head_dim):
    in_dim, out = 1536, 77
    W = qg.Int4Weight.from_numpy(I.int4_weight(5, I.TID_W, out, in_dim))
    y_in = qg.to_device(I.bf16_normal(5, I.TID_X, in_dim))
    z = qg.to_device(I.bf16_normal(6, I.TID_X, in_dim))
    gamma = qg.to_device(I.bf16_normal(7, I.TID_RESID, in_dim))
    out_b = Guarded(out, f32)
    ws = Guarded(qg.qg_workspace_bytes(qg.QG_OP_GATED_NORM, W, 0), u8)
    qg.gated_rmsnorm_qgemv_int4(W, y_in, z, gamma, 1e-6, head_dim, out=out_b.t, workspace=ws.t)
    _intact(out_b, ws)


def test_sigmoid_fma_guards(qg):
    out, in_dim = 33, 768
    W = qg.Int4Weight.from_numpy(I.int4_weight(8, I.TID_W, out, in_dim))
    gate = qg.to_device(np.array([0.3], np.float32))
    base = qg.to_device(I.f32_normal(8, I.TID_RESID, out))
    r = qg.to_device(I.bf16_normal(8, I.TID_RESID, out))
    y = Guarded(out, f32)
    qg.qgemv_int4_sigmoid_fma(W, qg.to_device(I.bf16_normal(8, I.TID_X, in_dim)), gate, base, r, y=y.t)
    o = Guarded(out, f32)
    qg.sigmoid_scalar_fma_residual(gate, base, base, r, out=o.t)
    _intact(y, o)


@pytest.mark.parametrize("E,hidden,inter,k", [(128, 2048, 768, 8), (9, 576, 128, 8), (5, 256, 192, 3), (4, 64, 64, 1)])
def test_moe_guards(qg, E, hidden, inter, k):
    gate = qg.Int4Weight.from_numpy(I.int4_weight(9, I.TID_GATE, inter, hidden, n_mat=E))
    up = qg.Int4Weight.from_numpy(I.int4_weight(9, I.TID_UP, inter, hidden, n_mat=E))
    down = qg.Int4Weight.from_numpy(I.int4_weight(9, I.TID_DOWN, hidden, inter, n_mat=E))
    logits = qg.to_device(I.f32_normal(9, I.TID_LOGITS, E))
    x = qg.to_device(I.bf16_normal(9, I.TID_X, hidden))
    r = qg.to_device(I.bf16_normal(9, I.TID_RESID, hidden))
    idx, p = Guarded(k, i32), Guarded(k, f32)
    qg.moe_router_topk(logits, k=k, idx=idx.t, p=p.t)
    y, ws = Guarded(hidden, f32), Guarded(qg.qg_workspace_bytes(qg.QG_OP_MOE, down, k), u8)
    qg.moe_gather_qgemv_int4(gate, up, down, idx.t, p.t, x, r, y=y.t, workspace=ws.t)
    y2, ws2 = Guarded(hidden, f32), Guarded(qg.qg_workspace_bytes(qg.QG_OP_MOE, down, k), u8)
    idx2, p2 = Guarded(k, i32), Guarded(k, f32)
    qg.moe_layer_int4(logits, gate, up, down, x, r, k=k, y=y2.t, idx=idx2.t, p=p2.t, workspace=ws2.t)
    v = qg.to_device(I.f32_normal(10, I.TID_X, (8, hidden)))
    c = Guarded(hidden, f32)
    qg.scalar_fma_chain8_residual(qg.to_device(I.f32_normal(10, I.TID_LOGITS, 8)), v, r, out=c.t)
    _intact(idx, p, y, ws, y2, ws2, idx2, p2, c)


@pytest.mark.parametrize("T,out,in_dim", [(1, 65, 128), (3, 100, 576), (8, 129, 1024), (17, 130, 1088),
                                          (33, 257, 2048), (257, 129, 192), (300, 200, 512)])
def test_qgemm_guards(qg, T, out, in_dim):
    W = qg.Int4Weight.from_numpy(I.int4_weight(11, I.TID_W, out, in_dim))
    X = qg.to_device(I.bf16_normal(11, I.TID_X, (T, in_dim)))
    Y = Guarded((T, out), f32)
    need = qg.qg_workspace_bytes(qg.QG_OP_QGEMM, W, T)
    ws = Guarded(max(need, 16), u8)
    qg.qgemm_int4(W, X, Y=Y.t, workspace=ws.t)
    outs = (out, 64, 1)
    Ws = [W] + [qg.Int4Weight.from_numpy(I.int4_weight(12, I.TID_MULTI + i, o, in_dim)) for i, o in enumerate(outs[1:])]
    Ys = [Guarded((T, o), f32) for o in outs]
    ws2 = Guarded(max(need, 16), u8)
    qg.qgemm_int4_multi(Ws, X, Ys=[y.t for y in Ys], workspace=ws2.t)
    _intact(Y, ws, ws2, *Ys)


@pytest.mark.parametrize("T", [1, 33, 257])
def test_moe_prefill_guards(qg, T):
    E, hidden, inter, k = 16, 512, 192, 4
    gate = qg.Int4Weight.from_numpy(I.int4_weight(13, I.TID_GATE, inter, hidden, n_mat=E))
    up = qg.Int4Weight.from_numpy(I.int4_weight(13, I.TID_UP, inter, hidden, n_mat=E))
    down = qg.Int4Weight.from_numpy(I.int4_weight(13, I.TID_DOWN, hidden, inter, n_mat=E))
    logits = qg.to_device(I.f32_normal(13, I.TID_LOGITS, (T, E)))
    X = qg.to_device(I.bf16_normal(13, I.TID_X, (T, hidden)))
    R = qg.to_device(I.bf16_normal(13, I.TID_RESID, (T, hidden)))
    Y, idx, p = Guarded((T, hidden), f32), Guarded((T, k), i32), Guarded((T, k), f32)
    ws = Guarded(qg.qg_workspace_bytes(qg.QG_OP_MOE_PREFILL, down, T), u8)
    qg.moe_prefill_int4(logits, gate, up, down, X, R, k=k, Y=Y.t, idx=idx.t, p=p.t, workspace=ws.t)
    _intact(Y, idx, p, ws)


@pytest.mark.parametrize("out,in_dim,bits", [(1, 64, 4), (33, 1088, 4), (7, 192, 2), (129, 576, 2)])
def test_quantize_guards(qg, out, in_dim, bits):
    w = qg.to_device(I.bf16_normal(14, I.TID_W, (out, in_dim)))
    packed = Guarded((out, in_dim * bits // 32), i32)
    scales, biases = Guarded((out, in_dim // 64), bf16), Guarded((out, in_dim // 64), bf16)
    rc = qg.lib.quantize_affine_q64a(qg._ptr(w), qg.QG_X_BF16, out, in_dim, bits, qg._ptr(packed.t),
                                     qg._ptr(scales.t), qg._ptr(biases.t), qg._stream(None))
    assert rc == qg.QG_OK
    _intact(packed, scales, biases)


@pytest.mark.parametrize("out,in_dim", [(1, 64), (33, 1088), (5121, 576)])
def test_q2_guards(qg, out, in_dim):
    d = I.int2_weight(15, I.TID_W, out, in_dim)
    t = qg.to_device
    W = qg.Int4Weight(t(d["packed"]), t(d["scales"]), t(d["biases"]), out, in_dim, bits=2)
    y = Guarded(out, f32)
    qg.qgemv_q2(W, t(I.bf16_normal(15, I.TID_X, in_dim)), y=y.t)
    _intact(y)

"""Degenerate cases of the decode path through the C ABI: a single expert slot (k = 1), every
expert selected (k = E), the router with n = k, an all-zero input vector (exactly zero output),
single-row outputs, and a one-row down projection after a layer."""
import numpy as np
import pytest

import oracle
from conftest import assert_within, assert_within_bound, dense_layer_reference
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _t(d):
    return (d["packed"], d["scales"], d["biases"])


@pytest.mark.parametrize("E,k", [(4, 1), (8, 8), (1, 1)])
def test_moe_single_slot_and_all_experts(qg, E, k):
    hidden, inter = 256, 128
    gate = I.int4_weight(E, I.TID_GATE, inter, hidden, n_mat=E)
    up = I.int4_weight(E, I.TID_UP, inter, hidden, n_mat=E)
    down = I.int4_weight(E, I.TID_DOWN, hidden, inter, n_mat=E)
    logits = I.f32_normal(E, I.TID_LOGITS, E)
    x = I.bf16_normal(E, I.TID_X, hidden)
    r = I.bf16_normal(E, I.TID_RESID, hidden)
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in (gate, up, down))
    y, idx, p = qg.moe_layer_int4(qg.to_device(logits), G, U, D, qg.to_device(x), qg.to_device(r), k=k)
    i_ref, p_ref = oracle.router_topk(logits, k)
    assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist()
    if k == E:
        assert sorted(i_ref.tolist()) == list(range(E))
    if k == 1:
        np.testing.assert_allclose(qg.to_numpy(p), [1.0], rtol=0, atol=0)
    y_ref, a, _ = oracle.moe(_t(gate), _t(up), _t(down), i_ref, p_ref, x, r)
    assert_within_bound(qg.to_numpy(y).astype(np.float64), y_ref, a)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_zero_input_gives_exact_zero(qg, kind):
    """x = 0: every group is dropped from the code term and the bias term is b * 0: y == 0."""
    d = I.int4_weight(1, I.TID_W, 300, 1024)
    x = np.zeros(1024, np.uint16 if kind == "bf16" else np.float32)
    y = qg.to_numpy(qg.qgemv_int4(qg.Int4Weight.from_numpy(d), qg.to_device(x)))
    assert np.all(y == 0.0)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("in_dim", [64, 5120, 17408])
def test_single_row_output(qg, in_dim):
    d = I.int4_weight(2, I.TID_W, 1, in_dim)
    x = I.bf16_normal(2, I.TID_X, in_dim)
    y = qg.to_numpy(qg.qgemv_int4(qg.Int4Weight.from_numpy(d), qg.to_device(x))).astype(np.float64)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    assert_within_bound(y, y_ref, a)


def test_layer_with_one_row_down(qg):
    """A layer whose down projection has a single output row (a scalar head after an FFN)."""
    g = I.int4_weight(3, I.TID_GATE, 640, 512)
    u = I.int4_weight(3, I.TID_UP, 640, 512)
    d = I.int4_weight(3, I.TID_DOWN, 1, 640)
    x = I.bf16_normal(3, I.TID_X, 512)
    G, U, D = (qg.Int4Weight.from_numpy(w) for w in (g, u, d))
    y = qg.to_numpy(qg.dense_layer_int4(G, U, D, qg.to_device(x))).astype(np.float64)
    # against the fp64 chain, within the bound propagated through SwiGLU and the down projection
    y_ref, y_bound, _, _ = dense_layer_reference(g, u, d, x)
    assert_within(y, y_ref, y_bound)


def test_router_n_equals_k(qg):
    logits = I.f32_normal(9, I.TID_LOGITS, 8)
    idx, p = qg.moe_router_topk(qg.to_device(logits), k=8)
    i_ref, p_ref = oracle.router_topk(logits, 8)
    assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist()
    np.testing.assert_allclose(qg.to_numpy(p), p_ref, rtol=2e-6, atol=1e-9)

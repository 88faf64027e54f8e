"""GPU parity of the MoE decode path (router, expert gather, chain8) against the fp64 oracle,
through the C ABI.  Router indices are compared bit-exactly; floating-point outputs against
|y - y_ref| <= 1e-3 * absref + 1e-6."""
import numpy as np
import pytest

import oracle
from conftest import assert_within_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _moe_weights(E, hidden, inter, seed=0):
    gate = I.int4_weight(seed, I.TID_GATE, inter, hidden, n_mat=E)
    up = I.int4_weight(seed, I.TID_UP, inter, hidden, n_mat=E)
    down = I.int4_weight(seed, I.TID_DOWN, hidden, inter, n_mat=E)
    return gate, up, down


def _t(d):
    return (d["packed"], d["scales"], d["biases"])


@pytest.fixture(scope="module")
def moe_full():
    """MoE decode T=1 at full size: hidden 2048, 128 experts, intermediate 768."""
    return _moe_weights(128, 2048, 768)


def test_router_pages_example(qg):
    logits = qg.to_device(np.array([1, 5, 3, 4], dtype=np.float32))
    idx, p = qg.moe_router_topk(logits, k=2)
    assert qg.to_numpy(idx).tolist() == [1, 3]
    np.testing.assert_allclose(qg.to_numpy(p), [0.7310585786300049, 0.2689414213699951], rtol=1e-6)


@pytest.mark.parametrize("n,k,renorm", [(128, 8, True), (128, 8, False), (1024, 32, True), (37, 5, True),
                                        (8, 8, True), (1, 1, True), (256, 8, False)])
def test_router_vs_oracle(qg, n, k, renorm):
    for seed in range(4):
        logits = I.f32_normal(seed, I.TID_LOGITS, n)
        idx, p = qg.moe_router_topk(qg.to_device(logits), k=k, renorm=renorm)
        i_ref, p_ref = oracle.router_topk(logits, k, renorm)
        assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist()
        np.testing.assert_allclose(qg.to_numpy(p), p_ref, rtol=2e-6, atol=1e-9)


def test_router_ties_take_lower_index(qg):
    logits = np.array([0.5, 2.0, -1.0, 2.0, 2.0, 0.0] + [2.0] * 40, dtype=np.float32)
    idx, _ = qg.moe_router_topk(qg.to_device(logits), k=5)
    assert qg.to_numpy(idx).tolist() == [1, 3, 4, 6, 7]


def _run_moe(qg, gate, up, down, idx_np, p_np, x, r):
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in (gate, up, down))
    idx = qg.to_device(idx_np.astype(np.uint32))
    p = qg.to_device(p_np.astype(np.float32))
    y = qg.moe_gather_qgemv_int4(G, U, D, idx, p, qg.to_device(x), qg.to_device(r))
    return qg.to_numpy(y).astype(np.float64)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_config3_moe_full(qg, moe_full, seed):
    """Router on the GPU, then the gather; compared with the oracle's router + MoE."""
    gate, up, down = moe_full
    logits = I.f32_normal(seed, I.TID_LOGITS, 128)
    x = I.bf16_normal(seed, I.TID_X, 2048)
    r = I.bf16_normal(seed, I.TID_RESID, 2048)
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in (gate, up, down))
    idx, p = qg.moe_router_topk(qg.to_device(logits), k=8)
    y = qg.moe_gather_qgemv_int4(G, U, D, idx, p, qg.to_device(x), qg.to_device(r))
    i_ref, p_ref = oracle.router_topk(logits, 8)
    assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist()
    y_ref, a, flags = oracle.moe(_t(gate), _t(up), _t(down), i_ref, p_ref, x, r)
    assert flags == 0
    assert_within_bound(qg.to_numpy(y).astype(np.float64), y_ref, a)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("E,hidden,inter,k", [(4, 128, 64, 2), (6, 576, 128, 8), (3, 1024, 192, 3),
                                              (16, 512, 768, 8)])
def test_moe_small_shapes(qg, E, hidden, inter, k):
    gate, up, down = _moe_weights(E, hidden, inter, seed=E)
    g = np.random.default_rng(E)
    idx = g.integers(0, E, k).astype(np.uint32)
    p = g.dirichlet(np.ones(k))
    x = I.bf16_normal(E, I.TID_X, hidden)
    r = I.bf16_normal(E, I.TID_RESID, hidden)
    y = _run_moe(qg, gate, up, down, idx, p, x, r)
    y_ref, a, _ = oracle.moe(_t(gate), _t(up), _t(down), idx, p.astype(np.float32).astype(np.float64), x, r)
    assert_within_bound(y, y_ref, a)


@pytest.mark.parametrize("e", [0, 63, 127])
def test_moe_one_hot_router_equals_single_expert(qg, moe_full, e):
    gate, up, down = moe_full
    idx = np.array([e, 1, 2, 3, 4, 5, 6, 7], dtype=np.uint32)
    p = np.array([1.0, 0, 0, 0, 0, 0, 0, 0])
    x = I.bf16_normal(9, I.TID_X, 2048)
    r = I.bf16_normal(9, I.TID_RESID, 2048)
    y = _run_moe(qg, gate, up, down, idx, p, x, r)
    y_ref, a, _ = oracle.moe(_t(gate), _t(up), _t(down), idx, p, x, r)
    assert_within_bound(y, y_ref, a)


def test_moe_bad_expert_index_is_skipped_and_flagged(qg):
    gate, up, down = _moe_weights(5, 256, 128, seed=11)
    idx = np.array([1, 77, 2, 3], dtype=np.uint32)
    p = np.full(4, 0.25)
    x = I.bf16_normal(11, I.TID_X, 256)
    r = I.bf16_normal(11, I.TID_RESID, 256)
    qg.qg_device_status()
    y = _run_moe(qg, gate, up, down, idx, p, x, r)
    assert qg.qg_device_status() & qg.QG_STATUS_BAD_EXPERT
    y_ref, a, flags = oracle.moe(_t(gate), _t(up), _t(down), idx, p, x, r)
    assert flags == 2
    assert_within_bound(y, y_ref, a)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("n", [2048, 2047, 5, 1, 4096 + 12])
def test_chain8(qg, n):
    p = np.array([0.3, 0.2, 0.15, 0.1, 0.1, 0.08, 0.05, 0.02], dtype=np.float32)
    v = I.f32_normal(n, 1, (8, n))
    r = I.bf16_normal(n, 2, n)
    out = qg.scalar_fma_chain8_residual(qg.to_device(p), qg.to_device(v), qg.to_device(r))
    y_ref, a = oracle.chain_residual(p.astype(np.float64), v, r)
    assert_within_bound(qg.to_numpy(out).astype(np.float64), y_ref, a)


def test_chain8_one_hot_is_exact(qg):
    n = 2048
    v = I.f32_normal(3, 1, (8, n))
    r = I.bf16_normal(3, 2, n)
    for k in range(8):
        p = np.zeros(8, dtype=np.float32)
        p[k] = 1.0
        out = qg.to_numpy(qg.scalar_fma_chain8_residual(qg.to_device(p), qg.to_device(v), qg.to_device(r)))
        np.testing.assert_array_equal(out, (I.bf16_bits_to_f32(r) + v[k]).astype(np.float32))


def test_router_signed_zero_and_negative_logits(qg):
    """-0.0 and +0.0 tie (the lower index wins); all-negative logits order by value."""
    logits = np.array([-0.0, 0.0, -1.0, -3.0, -0.5, 0.0, -2.0, -0.0], dtype=np.float32)
    idx, p = qg.moe_router_topk(qg.to_device(logits), k=4)
    i_ref, p_ref = oracle.router_topk(logits, 4)
    assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist() == [0, 1, 5, 7]
    np.testing.assert_allclose(qg.to_numpy(p), p_ref, rtol=2e-6)
    neg = -np.abs(I.f32_normal(3, I.TID_LOGITS, 300)) - 1.0
    idx, p = qg.moe_router_topk(qg.to_device(neg.astype(np.float32)), k=8, renorm=False)
    i_ref, p_ref = oracle.router_topk(neg.astype(np.float32), 8, False)
    assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist()
    np.testing.assert_allclose(qg.to_numpy(p), p_ref, rtol=2e-6, atol=1e-9)


@pytest.mark.parametrize("seed,renorm", [(0, True), (1, True), (2, False)])
def test_moe_layer_fused_router_matches_oracle_and_two_calls(qg, moe_full, seed, renorm):
    """moe_layer_int4 (router inside the gate/up kernel): indices bit-exact with the oracle's
    router, y within the bound, and the same result as moe_router_topk + moe_gather_qgemv_int4."""
    gate, up, down = moe_full
    logits = I.f32_normal(seed + 10, I.TID_LOGITS, 128)
    x = I.bf16_normal(seed + 10, I.TID_X, 2048)
    r = I.bf16_normal(seed + 10, I.TID_RESID, 2048)
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in (gate, up, down))
    lg, xd, rd = qg.to_device(logits), qg.to_device(x), qg.to_device(r)
    y, idx, p = qg.moe_layer_int4(lg, G, U, D, xd, rd, k=8, renorm=renorm)
    i_ref, p_ref = oracle.router_topk(logits, 8, renorm)
    assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist()
    np.testing.assert_allclose(qg.to_numpy(p), p_ref, rtol=2e-6, atol=1e-9)
    y_ref, a, flags = oracle.moe(_t(gate), _t(up), _t(down), i_ref, p_ref, x, r)
    assert flags == 0
    y_np = qg.to_numpy(y).astype(np.float64)
    assert_within_bound(y_np, y_ref, a)
    idx2, p2 = qg.moe_router_topk(lg, k=8, renorm=renorm)
    y2 = qg.to_numpy(qg.moe_gather_qgemv_int4(G, U, D, idx2, p2, xd, rd)).astype(np.float64)
    assert_within_bound(y_np, y2, 2 * a, what="fused vs two calls")
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("E,hidden,inter,k", [(4, 128, 64, 2), (9, 576, 128, 8), (37, 256, 192, 5),
                                           (300, 256, 64, 8), (1024, 128, 64, 7)])
def test_moe_layer_fused_small_shapes(qg, E, hidden, inter, k):
    """Both kernels select the experts themselves (more than 128 experts: keys re-read per round)."""
    gate, up, down = _moe_weights(E, hidden, inter, seed=E + 100)
    logits = I.f32_normal(E, I.TID_LOGITS, E)
    x = I.bf16_normal(E, I.TID_X, hidden)
    r = I.bf16_normal(E, I.TID_RESID, hidden)
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in (gate, up, down))
    y, idx, p = qg.moe_layer_int4(qg.to_device(logits), G, U, D, qg.to_device(x), qg.to_device(r), k=k)
    i_ref, p_ref = oracle.router_topk(logits, k)
    assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist()
    y_ref, a, _ = oracle.moe(_t(gate), _t(up), _t(down), i_ref, p_ref, x, r)
    assert_within_bound(qg.to_numpy(y).astype(np.float64), y_ref, a)


@pytest.mark.parametrize("E", [128, 200])
def test_moe_layer_fused_router_ties(qg, E):
    """Logits on a coarse grid (many ties): both kernels of the layer take the lower index first,
    as the oracle does, and agree with each other (y within the bound for the oracle's selection)."""
    hidden, inter, k = 256, 128, 8
    gate, up, down = _moe_weights(E, hidden, inter, seed=E + 7)
    logits = np.round(I.f32_normal(E + 7, I.TID_LOGITS, E) * 2.0).astype(np.float32) / 2.0
    x = I.bf16_normal(E + 7, I.TID_X, hidden)
    r = I.bf16_normal(E + 7, I.TID_RESID, hidden)
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in (gate, up, down))
    y, idx, p = qg.moe_layer_int4(qg.to_device(logits), G, U, D, qg.to_device(x), qg.to_device(r), k=k)
    i_ref, p_ref = oracle.router_topk(logits, k)
    assert len(set(logits[i_ref].tolist())) < k  # (the selection crosses a tie)
    assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist()
    y_ref, a, _ = oracle.moe(_t(gate), _t(up), _t(down), i_ref, p_ref, x, r)
    assert_within_bound(qg.to_numpy(y).astype(np.float64), y_ref, a)
    assert qg.qg_device_status() == 0

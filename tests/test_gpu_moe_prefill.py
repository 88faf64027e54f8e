"""GPU parity of moe_prefill_int4 (the MoE layer for T tokens: batched router, tokens grouped by
expert, grouped tensor-core gate/up and down, unpermuted weighted sum with the residual) against
the fp64 oracle applied token by token (router, expert gather, chain with residual).  Router
indices are compared bit for bit.  The projections run with fp16 operands, like qgemm_int4, so
the gate/up errors (within 1e-3 of their sum |w x|) reach y through SwiGLU and the down weights:
the bound adds 1e-3 * sum_s p_s sum_j |W_d[i][j]| dh_j, with dh the first-order SwiGLU bound of
the gate/up errors, to the oracle's 1e-3 * absref."""
import numpy as np
import pytest

import oracle
from conftest import ABS, REL, assert_within, assert_within_bound, swiglu_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _moe_weights(E, hidden, inter, seed=0):
    gate = I.int4_weight(seed, I.TID_GATE, inter, hidden, n_mat=E)
    up = I.int4_weight(seed, I.TID_UP, inter, hidden, n_mat=E)
    down = I.int4_weight(seed, I.TID_DOWN, hidden, inter, n_mat=E)
    return gate, up, down


def _t(d):
    return (d["packed"], d["scales"], d["biases"])


def _expert(d, e):
    return tuple(np.ascontiguousarray(a[e]) for a in _t(d))


def _check_token(ws, logits_t, x_t, r_t, k, renorm, y_t, idx_t):
    """One token: indices bit-exact; y against the oracle's MoE (h in fp64) within the bound of the
    down GEMVs on the GPU's h (1e-3 sum |w h~| + 1e-6) plus the gate/up errors carried through
    SwiGLU and the down weights: |y~ - y| <= 1e-3 (A + D) + 1e-6 + D, D = sum_s p_s sum_j
    |W_d[e_s][i][j]| dh_s[j] (conftest.swiglu_bound; the route weights are exact inputs to both)."""
    gate, up, down = ws
    i_ref, p_ref = oracle.router_topk(logits_t, k, renorm)
    assert idx_t.tolist() == i_ref.tolist()
    y_ref, a, flags = oracle.moe(_t(gate), _t(up), _t(down), i_ref, p_ref, x_t, r_t)
    assert flags == 0
    extra = np.zeros_like(a)
    for s, e in enumerate(i_ref.tolist()):
        g, ag = oracle.qgemv(*_expert(gate, e), x_t)
        u, au = oracle.qgemv(*_expert(up, e), x_t)
        _, dab = oracle.qgemv_f64x(*_expert(down, e), swiglu_bound(g, u, REL * ag + ABS, REL * au + ABS))
        extra += abs(p_ref[s]) * dab
    assert_within(y_t, y_ref, REL * (a + extra) + ABS + extra)


def _run(qg, ws, T, k, renorm=True, residual=True, seed=0):
    E = ws[0]["packed"].shape[0]
    hidden = ws[0]["packed"].shape[2] * 8
    logits = I.f32_normal(seed, I.TID_LOGITS, (T, E))
    X = I.bf16_normal(seed, I.TID_X, (T, hidden))
    R = I.bf16_normal(seed, I.TID_RESID, (T, hidden)) if residual else np.zeros((T, hidden), np.uint16)
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in ws)
    Y, idx, p = qg.moe_prefill_int4(qg.to_device(logits), G, U, D, qg.to_device(X),
                                    qg.to_device(R) if residual else None, k=k, renorm=renorm)
    assert qg.qg_device_status() == 0
    return logits, X, R, qg.to_numpy(Y).astype(np.float64), qg.to_numpy(idx).astype(np.uint32), qg.to_numpy(p)


@pytest.mark.parametrize("E,hidden,inter,T,k", [
    (8, 256, 128, 37, 2),      # a few tokens per expert, one tile each
    (4, 128, 64, 300, 2),      # 150 rows per expert: two 128-row tiles per expert
    (64, 512, 256, 3, 8),      # most experts empty
    (16, 384, 192, 50, 1),     # k = 1
])
def test_moe_prefill_small_shapes(qg, E, hidden, inter, T, k):
    ws = _moe_weights(E, hidden, inter, seed=E + T)
    logits, X, R, Y, idx, p = _run(qg, ws, T, k, seed=T)
    for t in range(T):
        _check_token(ws, logits[t], X[t], R[t], k, True, Y[t], idx[t])


@pytest.mark.parametrize("renorm", [True, False])
def test_moe_prefill_no_residual_and_softmax_modes(qg, renorm):
    ws = _moe_weights(8, 256, 128, seed=5)
    logits, X, R, Y, idx, p = _run(qg, ws, 20, 4, renorm=renorm, residual=False, seed=5)
    for t in range(20):
        _check_token(ws, logits[t], X[t], R[t], 4, renorm, Y[t], idx[t])
        _, p_ref = oracle.router_topk(logits[t], 4, renorm)
        np.testing.assert_allclose(p[t], p_ref, rtol=1e-5, atol=1e-7)


@pytest.fixture(scope="module")
def moe_full():
    """The MoE config's shapes: 128 experts, hidden 2048, intermediate 768."""
    return _moe_weights(128, 2048, 768)


@pytest.mark.parametrize("T", [256, 33])
def test_moe_prefill_full_size_sampled_tokens(qg, moe_full, T):
    """T tokens over 128 experts (top 8): indices of every token bit-exact, y of sampled tokens."""
    logits, X, R, Y, idx, p = _run(qg, moe_full, T, 8, seed=T)
    for t in range(T):
        i_ref, _ = oracle.router_topk(logits[t], 8)
        assert idx[t].tolist() == i_ref.tolist(), t
    rng = np.random.default_rng(T)
    for t in sorted(set([0, T - 1] + rng.integers(0, T, 4).tolist())):
        _check_token(moe_full, logits[t], X[t], R[t], 8, True, Y[t], idx[t])


def test_moe_prefill_rejects_bad_arguments(qg):
    import torch

    ws = _moe_weights(8, 256, 128, seed=1)
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in ws)
    X = qg.to_device(I.bf16_normal(1, I.TID_X, (4, 256)))
    logits = qg.to_device(I.f32_normal(1, I.TID_LOGITS, (4, 8)))
    with pytest.raises(qg.QGError) as e:
        qg.moe_prefill_int4(logits, G, U, D, X, k=9)
    assert e.value.code == qg.QG_EINVAL
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(qg.QGError) as e:
        qg.moe_prefill_int4(logits, G, U, D, X, k=2, workspace=small)
    assert e.value.code == qg.QG_EWORKSPACE
    assert qg.qg_device_status() == 0


def test_moe_prefill_is_deterministic(qg, moe_full):
    """The plan places rows within an expert's group in atomic order, which may differ from call to
    call; every row is computed independently of its neighbours, so y, indices and weights are bit
    for bit the same over repeated calls."""
    T = 64
    logits = qg.to_device(I.f32_normal(3, I.TID_LOGITS, (T, 128)))
    X = qg.to_device(I.bf16_normal(3, I.TID_X, (T, 2048)))
    R = qg.to_device(I.bf16_normal(3, I.TID_RESID, (T, 2048)))
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in moe_full)
    first = [qg.to_numpy(a) for a in qg.moe_prefill_int4(logits, G, U, D, X, R, k=8)]
    for _ in range(3):
        again = [qg.to_numpy(a) for a in qg.moe_prefill_int4(logits, G, U, D, X, R, k=8)]
        for a, b in zip(first, again):
            np.testing.assert_array_equal(a, b)
    assert qg.qg_device_status() == 0

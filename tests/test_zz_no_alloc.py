"""moe_gather_qgemv_int4_noalloc (the MoE gather step on the library's fixed scratch) against the
workspace entry point moe_gather_qgemv_int4 and the fp64 oracle, on two calls in a row.

Named to be collected last, so it runs both after the rest of the GPU suite and, alone, in a fresh
process (the first call there does the per-device address lookup)."""
import numpy as np
import pytest

import oracle
from conftest import assert_within_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _t(d):
    return (d["packed"], d["scales"], d["biases"])


def _weights(E, hidden, inter, seed):
    gate = I.int4_weight(seed, I.TID_GATE, inter, hidden, n_mat=E)
    up = I.int4_weight(seed, I.TID_UP, inter, hidden, n_mat=E)
    down = I.int4_weight(seed, I.TID_DOWN, hidden, inter, n_mat=E)
    return gate, up, down


def _two_calls(qg, E, hidden, inter, k, seed):
    import torch

    gate, up, down = _weights(E, hidden, inter, seed)
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in (gate, up, down))
    # inputs and outputs of both calls exist before the first no-alloc call
    cases = []
    for c in range(2):
        g = np.random.default_rng([seed, c])
        idx = g.choice(E, size=k, replace=False).astype(np.uint32) if k <= E else g.integers(0, E, k).astype(np.uint32)
        p = g.dirichlet(np.ones(k)).astype(np.float32)
        x = I.bf16_normal(seed + c, I.TID_X, hidden)
        r = I.bf16_normal(seed + c, I.TID_RESID, hidden)
        dev = [qg.to_device(a) for a in (idx, p, x, r)]
        cases.append((idx, p, x, r, dev, torch.full((hidden,), float("nan"), device="cuda")))
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    for idx, p, x, r, (di, dp, dx, dr), y in cases:
        qg.moe_gather_qgemv_int4_noalloc(G, U, D, di, dp, dx, dr, y)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before
    for idx, p, x, r, (di, dp, dx, dr), y in cases:
        y_ws = qg.moe_gather_qgemv_int4(G, U, D, di, dp, dx, dr)
        y_ref, a, flags = oracle.moe(_t(gate), _t(up), _t(down), idx, p.astype(np.float64), x, r)
        assert flags == 0
        y_na = qg.to_numpy(y).astype(np.float64)
        assert_within_bound(y_na, qg.to_numpy(y_ws).astype(np.float64), a, what="noalloc vs workspace")
        assert_within_bound(y_na, y_ref, a, what="noalloc vs oracle")
    assert qg.qg_device_status() == 0


def test_noalloc_moe_decode_two_calls(qg):
    """MoE decode T=1: hidden 2048, 128 experts, intermediate 768, top-8."""
    _two_calls(qg, 128, 2048, 768, 8, seed=21)


def test_noalloc_at_scratch_limit_two_calls(qg):
    """k * inter exactly at the fixed scratch size (8 x 4096 fp32)."""
    assert 8 * 4096 == qg.QG_NOALLOC_MOE_MAX_FLOATS
    _two_calls(qg, 8, 256, 4096, 8, seed=22)


def test_noalloc_small_ragged(qg):
    _two_calls(qg, 6, 576, 128, 3, seed=23)


def test_noalloc_rejects_over_limit(qg):
    import torch

    gate, up, down = _weights(1, 64, 4160, seed=24)
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in (gate, up, down))
    idx = qg.to_device(np.zeros(8, dtype=np.uint32))
    p = qg.to_device(np.full(8, 0.125, dtype=np.float32))
    x = qg.to_device(I.bf16_normal(24, I.TID_X, 64))
    r = qg.to_device(I.bf16_normal(24, I.TID_RESID, 64))
    y = torch.zeros(64, device="cuda")
    with pytest.raises(qg.QGError) as e:
        qg.moe_gather_qgemv_int4_noalloc(G, U, D, idx, p, x, r, y)
    assert e.value.code == qg.QG_ENOTSUP
    assert torch.count_nonzero(y).item() == 0

"""GPU parity of qgemm_int4 (T token rows) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from conftest import assert_within_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _run(qg, d, X):
    Y = qg.qgemm_int4(qg.Int4Weight.from_numpy(d), qg.to_device(X))
    return qg.to_numpy(Y).astype(np.float64)


@pytest.mark.parametrize("T,out,in_dim", [(1, 64, 128), (3, 100, 576), (8, 300, 1024), (33, 256, 2048),
                                          (40, 130, 1088)])
def test_qgemm_small(qg, T, out, in_dim):
    d = I.int4_weight(T, I.TID_W, out, in_dim)
    X = I.bf16_normal(T, I.TID_X, (T, in_dim))
    Y = _run(qg, d, X)
    Y_ref, A = oracle.qgemm(d["packed"], d["scales"], d["biases"], X)
    assert_within_bound(Y, Y_ref, A)


@pytest.mark.parametrize("T", [8, 32, 256])
def test_config4_full_size_sampled_rows(qg, T):
    """W 17408 x 5120, X T x 5120: every token row, 48 sampled output rows."""
    d = I.int4_weight(0, I.TID_W, 17408, 5120)
    X = I.bf16_normal(0, I.TID_X, (T, 5120))
    Y = _run(qg, d, X)
    g = np.random.default_rng(T)
    for r in sorted(set([0, 17407, 8704] + list(g.integers(0, 17408, 45)))):
        Yr, Ar = oracle.qgemm(d["packed"], d["scales"], d["biases"], X, rows=(r, r + 1))
        assert_within_bound(Y[:, r:r + 1], Yr, Ar, what=f"row {r}")

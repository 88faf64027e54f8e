"""GPU parity of qgemm_int4 (T token rows) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from conftest import ORACLE_THREADS, assert_within_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _run(qg, d, X):
    Y = qg.qgemm_int4(qg.Int4Weight.from_numpy(d), qg.to_device(X))
    return qg.to_numpy(Y).astype(np.float64)


@pytest.mark.parametrize("T,out,in_dim", [(1, 64, 128), (3, 100, 576), (8, 300, 1024), (33, 256, 2048),
                                          (40, 130, 1088), (20, 129, 512), (57, 140, 1536), (64, 200, 1024)])
def test_qgemm_small(qg, T, out, in_dim):
    """Ragged rows and token counts; in a multiple of 512 with T <= 64 is the small-tile tensor-copy
    kernel (two MMA-issuing threads, two accumulators) at every tile height from 16 to 64."""
    d = I.int4_weight(T, I.TID_W, out, in_dim)
    X = I.bf16_normal(T, I.TID_X, (T, in_dim))
    Y = _run(qg, d, X)
    Y_ref, A = oracle.qgemm(d["packed"], d["scales"], d["biases"], X)
    assert_within_bound(Y, Y_ref, A)


@pytest.mark.parametrize("T", [8, 32, 256])
def test_config4_full_size(qg, T):
    """W 17408 x 5120, X T x 5120, in the default dispatch: every row of every token for T = 8 and
    32; for T = 256 every row of four tokens (the first and last of each 128-token half) and every
    token of two rows of each 128-row tile, so every (row tile, token tile) pair is checked."""
    d = I.int4_weight(0, I.TID_W, 17408, 5120)
    X = I.bf16_normal(0, I.TID_X, (T, 5120))
    Y = _run(qg, d, X)
    if T <= 32:
        Y_ref, A = oracle.qgemm(d["packed"], d["scales"], d["biases"], X, threads=ORACLE_THREADS)
        assert_within_bound(Y, Y_ref, A)
        return
    for t in (0, 127, 128, 255):
        yr, ar = oracle.qgemv(d["packed"], d["scales"], d["biases"], X[t], threads=ORACLE_THREADS)
        assert_within_bound(Y[t], yr, ar, what=f"token {t}")
    for r0 in range(0, 17408, 128):
        for r in (r0 + 5, r0 + 122):
            Yr, Ar = oracle.qgemm(d["packed"], d["scales"], d["biases"], X, rows=(r, r + 1))
            assert_within_bound(Y[:, r:r + 1], Yr, Ar, what=f"row {r}")


@pytest.mark.parametrize("in_dim,T", [(17408, 32), (17408, 256), (32768, 48)])
def test_qgemm_tensor_core_long_k(qg, in_dim, T):
    """The tensor-core path at the down projection's K = 17408 (and the largest K, 32768): the
    fp32 accumulation over 1088 (2048) MMA steps stays within the bound (every row, every token)."""
    out = 640
    d = I.int4_weight(in_dim, I.TID_W, out, in_dim)
    X = I.bf16_normal(in_dim, I.TID_X, (T, in_dim))
    Y = _run(qg, d, X)
    Y_ref, A = oracle.qgemm(d["packed"], d["scales"], d["biases"], X, threads=ORACLE_THREADS)
    assert_within_bound(Y, Y_ref, A)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("T,out,in_dim", [(16, 128, 64), (32, 128, 128), (48, 130, 1088), (256, 384, 2048),
                                          (300, 200, 512), (257, 129, 192)])
def test_qgemm_tensor_core_shapes(qg, T, out, in_dim):
    """The tensor-core path (the threshold forced to 16): one and several token tiles, ragged rows."""
    qg.qg_tune_qgemm(16)
    try:
        d = I.int4_weight(T + 7, I.TID_W, out, in_dim)
        X = I.bf16_normal(T + 7, I.TID_X, (T, in_dim))
        Y = _run(qg, d, X)
    finally:
        qg.qg_tune_qgemm(0)
    Y_ref, A = oracle.qgemm(d["packed"], d["scales"], d["biases"], X)
    assert_within_bound(Y, Y_ref, A)
    assert qg.qg_device_status() == 0


def test_qgemm_t8_tensor_core_matches_gemv_path(qg):
    """T = 8 padded onto the tensor cores equals the CUDA-core GEMV path within the bound."""
    d = I.int4_weight(8, I.TID_W, 640, 1024)
    X = I.bf16_normal(8, I.TID_X, (8, 1024))
    qg.qg_tune_qgemm(9)  # T = 8 below the threshold: the per-token GEMV path
    try:
        y_gemv = _run(qg, d, X)
    finally:
        qg.qg_tune_qgemm(0)
    y_tc = _run(qg, d, X)  # the default for T = 8: the tensor cores
    Y_ref, A = oracle.qgemm(d["packed"], d["scales"], d["biases"], X)
    assert_within_bound(y_gemv, Y_ref, A, what="gemv path")
    assert_within_bound(y_tc, Y_ref, A, what="tensor-core path")
    assert_within_bound(y_tc, y_gemv, 2 * A, what="tensor core vs gemv")


def test_qgemm_token_scales_extreme_rows(qg):
    """Token rows of very different magnitudes (one all zero) keep the per-row bound on the tensor cores."""
    T, out, in_dim = 32, 256, 512
    d = I.int4_weight(5, I.TID_W, out, in_dim)
    x = I.bf16_normal(5, I.TID_X, (T, in_dim)).astype(np.uint32)
    f = (x << 16).view(np.float32).astype(np.float64)
    f[1] *= 2.0 ** 40
    f[2] *= 2.0 ** -40
    f[3] = 0.0
    X = I.f64_to_bf16_bits(f).reshape(T, in_dim)
    Y = _run(qg, d, X)
    Y_ref, A = oracle.qgemm(d["packed"], d["scales"], d["biases"], X)
    assert_within_bound(Y, Y_ref, A)
    assert np.all(Y[3] == 0.0)


def _multi(qg, outs, in_dim, T, seed):
    ds = [I.int4_weight(seed, I.TID_MULTI + i, o, in_dim) for i, o in enumerate(outs)]
    X = I.bf16_normal(seed, I.TID_X, (T, in_dim))
    Ys = qg.qgemm_int4_multi([qg.Int4Weight.from_numpy(d) for d in ds], qg.to_device(X))
    return ds, X, [qg.to_numpy(Y).astype(np.float64) for Y in Ys]


@pytest.mark.parametrize("outs,in_dim,T", [((8192, 4096, 32, 32), 2048, 256), ((8192, 4096, 32, 32), 2048, 8),
                                           ((4096, 512, 512), 2048, 100), ((200, 64), 576, 33),
                                           ((130, 260, 1), 1088, 300)])
def test_qgemm_multi_vs_oracle(qg, outs, in_dim, T):
    """Prefill form of the shared-input projections (quartet / triple of config 2, and ragged
    sets): every row of every matrix against the oracle, every token."""
    ds, X, Ys = _multi(qg, outs, in_dim, T, seed=T + len(outs))
    for d, Y, o in zip(ds, Ys, outs):
        assert Y.shape == (T, o)
        Yr, Ar = oracle.qgemm(d["packed"], d["scales"], d["biases"], X, threads=ORACLE_THREADS)
        assert_within_bound(Y, Yr, Ar)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("T", [8, 64])
def test_qgemm_multi_equals_separate_calls(qg, T):
    """One launch over all matrices gives bit for bit what one qgemm_int4 call per matrix gives."""
    outs = (1000, 300, 64)
    ds, X, Ys = _multi(qg, outs, 1024, T, seed=77)
    for d, Y in zip(ds, Ys):
        np.testing.assert_array_equal(Y, _run(qg, d, X))

"""GPU parity of qgemv_int4 / qgemv_int4_multi against the fp64 oracle, through the C ABI.

Bound (every fp32 output): |y - y_ref| <= 1e-3 * sum|w*x| + 1e-6, with y_ref and sum|w*x| from the
oracle on the same stored inputs.  Nibble decoding is checked bit-exactly with one-hot inputs."""
import math

import numpy as np
import pytest

import oracle
from conftest import ABS, ORACLE_THREADS, REL, assert_within, assert_within_bound, swiglu_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _run_gemv(qg, d, x_np, xf32=False):
    w = qg.Int4Weight.from_numpy(d)
    x = qg.to_device(x_np)
    y = qg.qgemv_int4(w, x)
    return qg.to_numpy(y).astype(np.float64)


# shapes spanning several stages and CTAs, ragged tails, and the non-bulk scale path (in % 512 != 0)
SHAPES = [(1, 64), (7, 64), (33, 128), (77, 576), (256, 1024), (300, 1088), (1000, 2048), (513, 4160),
          (2049, 512), (40, 11264), (24, 32768)]


@pytest.mark.parametrize("out,in_dim", SHAPES)
def test_qgemv_bf16_small_shapes(qg, out, in_dim):
    d = I.int4_weight(0, I.TID_W, out, in_dim)
    x = I.bf16_normal(0, I.TID_X, in_dim)
    y = _run_gemv(qg, d, x)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    assert_within_bound(y, y_ref, a)


@pytest.mark.parametrize("out,in_dim", [(5, 64), (77, 576), (300, 1088), (129, 17408)])
def test_qgemv_f32_input(qg, out, in_dim):
    d = I.int4_weight(1, I.TID_W, out, in_dim)
    x = I.f32_normal(1, I.TID_X, in_dim) * np.float32(3.7)
    y = _run_gemv(qg, d, x)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    assert_within_bound(y, y_ref, a)


def test_config0_full(qg):
    """int4 affine dequant-GEMV M=1, W 256 x 1024, seed 0: every row."""
    d = I.int4_weight(0, I.TID_W, 256, 1024)
    x = I.bf16_normal(0, I.TID_X, 1024)
    y = _run_gemv(qg, d, x)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    assert_within_bound(y, y_ref, a)


@pytest.mark.parametrize("j", [0, 1, 2, 3, 4, 5, 6, 7, 31, 32, 63, 64, 65, 511, 512, 1023])
def test_one_hot_x_decodes_nibbles_exactly(qg, j):
    """x = e_j makes y[r] = fp32(scale * q[r][j] + bias): equal bit for bit to the oracle's value
    rounded to fp32, for every row, so every nibble position and group edge is decoded exactly."""
    d = I.int4_weight(2, I.TID_W, 96, 1024, keep_codes=True)
    x = np.zeros(1024, dtype=np.uint16)
    x[j] = 0x3F80
    y = qg.to_numpy(qg.qgemv_int4(qg.Int4Weight.from_numpy(d), qg.to_device(x)))
    y_ref, _ = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    np.testing.assert_array_equal(y, y_ref.astype(np.float32))


def test_all_zero_codes(qg):
    d = I.int4_weight(3, I.TID_W, 130, 2048)
    d["packed"] = np.zeros_like(d["packed"])
    x = I.bf16_normal(3, I.TID_X, 2048)
    y = _run_gemv(qg, d, x)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    assert_within_bound(y, y_ref, a)


def test_extreme_x_ranges(qg):
    """Large and tiny input magnitudes in one vector (per-unit power-of-two scaling)."""
    d = I.int4_weight(4, I.TID_W, 64, 1024)
    g = np.random.default_rng(4)
    x64 = g.standard_normal(1024) * np.exp2(g.integers(-30, 30, 1024))
    x64[100:132] = 0.0
    x64[200:232] *= 1e-12
    x = I.f64_to_bf16_bits(x64)
    y = _run_gemv(qg, d, x)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    assert_within_bound(y, y_ref, a)


@pytest.mark.parametrize("out,in_dim", [(17408, 5120), (5120, 17408)])
def test_config1_full_size_every_row(qg, out, in_dim):
    """Dense decode projections at full size (gate/up 17408 x 5120, down 5120 x 17408), in the
    launch configuration the benchmark times (PDL on): every row against the oracle."""
    d = I.int4_weight(0, I.TID_GATE if out == 17408 else I.TID_DOWN, out, in_dim)
    x = I.bf16_normal(0, I.TID_X, in_dim)
    prev = qg.qg_set_pdl(True)
    try:
        y = _run_gemv(qg, d, x)
    finally:
        qg.qg_set_pdl(prev)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x, threads=ORACLE_THREADS)
    assert_within_bound(y, y_ref, a)


def _multi(qg, outs, in_dim, seed=0):
    ds = [I.int4_weight(seed, I.TID_MULTI + i, o, in_dim) for i, o in enumerate(outs)]
    x = I.bf16_normal(seed, I.TID_X, in_dim)
    ws = [qg.Int4Weight.from_numpy(d) for d in ds]
    ys = qg.qgemv_int4_multi(ws, qg.to_device(x))
    return ds, x, [qg.to_numpy(y).astype(np.float64) for y in ys]


@pytest.mark.parametrize("outs", [(8192, 4096, 32, 32), (4096, 512, 512)])
def test_config2_multi_full(qg, outs):
    """Shared-input multi-projection GEMV, in=2048: the qkv/z/b/a quartet and the 3-way variant."""
    ds, x, ys = _multi(qg, outs, 2048)
    for d, y in zip(ds, ys):
        y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
        assert_within_bound(y, y_ref, a)


@pytest.mark.parametrize("outs,in_dim", [((3, 5), 64), ((100, 1, 37), 576), ((16, 16, 16, 16), 1024)])
def test_multi_ragged(qg, outs, in_dim):
    ds, x, ys = _multi(qg, outs, in_dim, seed=5)
    for d, y in zip(ds, ys):
        y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
        assert_within_bound(y, y_ref, a)


def test_multi_equals_separate_calls(qg):
    ds, x, ys = _multi(qg, (8192, 4096, 32, 32), 2048, seed=6)
    for d, y in zip(ds, ys):
        np.testing.assert_array_equal(y, _run_gemv(qg, d, x))


@pytest.mark.parametrize("out,in_dim", [(40, 128), (1000, 576), (17408, 5120)])
def test_swiglu_pair(qg, out, in_dim):
    """h = silu(W_g x) * (W_u x) in one launch, every row, within the GEMV bounds on g and u carried
    through SwiGLU (conftest.swiglu_bound)."""
    gd = I.int4_weight(0, I.TID_GATE, out, in_dim)
    ud = I.int4_weight(0, I.TID_UP, out, in_dim)
    x = I.bf16_normal(0, I.TID_X, in_dim)
    h = qg.qgemv_int4_multi([qg.Int4Weight.from_numpy(gd), qg.Int4Weight.from_numpy(ud)], qg.to_device(x),
                            epilogue="swiglu")
    h = qg.to_numpy(h).astype(np.float64)
    g, ag = oracle.qgemv(gd["packed"], gd["scales"], gd["biases"], x, threads=ORACLE_THREADS)
    u, au = oracle.qgemv(ud["packed"], ud["scales"], ud["biases"], x, threads=ORACLE_THREADS)
    assert_within(h, oracle.swiglu(g, u), swiglu_bound(g, u, REL * ag + ABS, REL * au + ABS))


def test_pdl_and_determinism(qg):
    d = I.int4_weight(0, I.TID_W, 5120, 4096)
    x = I.bf16_normal(0, I.TID_X, 4096)
    y0 = _run_gemv(qg, d, x)
    prev = qg.qg_set_pdl(True)
    try:
        w = qg.Int4Weight.from_numpy(d)
        xd = qg.to_device(x)
        ys = [qg.to_numpy(qg.qgemv_int4(w, xd)) for _ in range(3)]
    finally:
        qg.qg_set_pdl(prev)
    for y in ys:
        np.testing.assert_array_equal(y.astype(np.float64), y0)
    assert qg.qg_device_status() == 0


def test_device_wait_timeout_sets_status_and_context_survives(qg):
    """A device wait that nothing completes gives up after its limit, sets QG_STATUS_TIMEOUT and the
    context stays usable for the next call."""
    import torch

    qg.qg_device_status()  # clear
    qg.qg_selftest_wait_timeout(2000)
    torch.cuda.synchronize()
    assert qg.qg_device_status() & qg.QG_STATUS_TIMEOUT
    assert qg.qg_device_status() == 0  # read-and-clear
    d = I.int4_weight(1, I.TID_W, 64, 128)
    x = I.bf16_normal(1, I.TID_X, 128)
    y = qg.to_numpy(qg.qgemv_int4(qg.Int4Weight.from_numpy(d), qg.to_device(x))).astype(np.float64)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    assert_within_bound(y, y_ref, a)
    assert qg.qg_device_status() == 0
    with pytest.raises(qg.QGError):
        qg.qg_selftest_wait_timeout(0)

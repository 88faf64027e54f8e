"""Inputs with outlier channels, through the C ABI against the fp64 oracle.

Activations of real models carry a few channels 10^3 - 10^4 times larger than the rest.  In a
64-column group holding such a channel, a single 16-bit fixed-point pass scaled to the outlier
leaves the other entries with a few bits; when the outlier meets a zero weight, nothing in the row
is large enough to hide that error.  The GEMV takes a second 16-bit pass for such groups (a numpy
emulation of the one-pass kernel misses the bound of the first case's lone group by a factor of
about 400)."""
import numpy as np
import pytest

import oracle
from conftest import ABS, ORACLE_THREADS, REL, assert_within, assert_within_bound, dense_layer_reference, swiglu_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu

OUTLIERS = {5: 1.0e3, 700: -3.0e3, 1029: 1.0e4, 3000: -6.5e3}  # channel -> value (rounded to bf16)
ZERO_CH = 1029  # the outlier that sits on an exactly-zero weight in every other row


def _set_codes(d, rows, col, code):
    """Set the 4-bit code of (row, col) for every row in `rows` (packed u32, low nibble first)."""
    w, sh = col // 8, 4 * (col % 8)
    for r in rows:
        d["packed"][r, w] = (d["packed"][r, w] & ~np.uint32(0xF << sh)) | np.uint32(code << sh)


def _zero_weight(d, rows, col):
    """w[r][col] = s * 8 + b = 0 exactly: code 8 and b = -8 s (exact in bf16: a power-of-two
    multiple of the bf16 scale)."""
    _set_codes(d, rows, col, 8)
    g = col // 64
    s = I.bf16_bits_to_f32(d["scales"][rows, g]).astype(np.float64)
    d["biases"][rows, g] = I.f64_to_bf16_bits(-8.0 * s)


def _x_with_outliers(seed, n, kind="bf16"):
    x = I.rng(seed, I.TID_X).standard_normal(n)
    for c, v in OUTLIERS.items():
        if c < n:
            x[c] = v
    return I.f64_to_bf16_bits(x) if kind == "bf16" else x.astype(np.float32)


def _w_with_zeros(seed, tid, out, in_dim, n_mat=None):
    d = I.int4_weight(seed, tid, out, in_dim, n_mat=n_mat)
    if ZERO_CH < in_dim:
        if n_mat is None:
            _zero_weight(d, np.arange(0, out, 2), ZERO_CH)
        else:
            for e in range(n_mat):
                sub = {k: v[e] for k, v in d.items()}
                _zero_weight(sub, np.arange(0, out, 2), ZERO_CH)
    return d


def test_single_outlier_on_zero_weight_group(qg):
    """The worked case: one group holds x0 = 2^10 on a zero weight (code 8, bias -8 s) and 63
    entries of 2^-6; a first pass scaled to 2^10 rounds all 63 to zero.  Every row is checked."""
    out, in_dim = 96, 256
    d = I.int4_weight(21, I.TID_W, out, in_dim)
    _zero_weight(d, np.arange(out), 64)
    x = np.full(in_dim, 2.0 ** -6)
    x[64] = 2.0 ** 10
    x[:64] = I.rng(21, I.TID_X).standard_normal(64)
    x[128:] = I.rng(22, I.TID_X).standard_normal(128)
    xb = I.f64_to_bf16_bits(x)
    y = qg.to_numpy(qg.qgemv_int4(qg.Int4Weight.from_numpy(d), qg.to_device(xb))).astype(np.float64)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], xb)
    assert_within_bound(y, y_ref, a)
    # the group on its own (the other groups' x zero): the row is all in the small entries
    x2 = np.zeros(in_dim)
    x2[64:128] = x[64:128]
    xb2 = I.f64_to_bf16_bits(x2)
    y2 = qg.to_numpy(qg.qgemv_int4(qg.Int4Weight.from_numpy(d), qg.to_device(xb2))).astype(np.float64)
    y2_ref, a2 = oracle.qgemv(d["packed"], d["scales"], d["biases"], xb2)
    assert_within_bound(y2, y2_ref, a2)


@pytest.mark.parametrize("out,in_dim", [(5120, 17408), (2048, 4096), (300, 1088)])
@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_qgemv_outlier_channels(qg, out, in_dim, kind):
    d = _w_with_zeros(31, I.TID_W, out, in_dim)
    x = _x_with_outliers(31, in_dim, kind)
    y = qg.to_numpy(qg.qgemv_int4(qg.Int4Weight.from_numpy(d), qg.to_device(x))).astype(np.float64)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x, threads=ORACLE_THREADS)
    assert_within_bound(y, y_ref, a)
    assert qg.qg_device_status() == 0


def test_multi_and_pair_outlier_channels(qg):
    """The shared-input quartet and the SwiGLU pair with outlier channels in x."""
    outs = (8192, 4096, 32, 32)
    ds = [_w_with_zeros(41, I.TID_MULTI + i, o, 2048) for i, o in enumerate(outs)]
    x = _x_with_outliers(41, 2048)
    ys = qg.qgemv_int4_multi([qg.Int4Weight.from_numpy(d) for d in ds], qg.to_device(x))
    for d, y in zip(ds, ys):
        y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x, threads=ORACLE_THREADS)
        assert_within_bound(qg.to_numpy(y).astype(np.float64), y_ref, a)
    g, u = ds[0], ds[1]
    g = _w_with_zeros(42, I.TID_GATE, 4096, 2048)
    h = qg.qgemv_int4_multi([qg.Int4Weight.from_numpy(g), qg.Int4Weight.from_numpy(u)], qg.to_device(x),
                            epilogue="swiglu")
    gr, ag = oracle.qgemv(g["packed"], g["scales"], g["biases"], x, threads=ORACLE_THREADS)
    ur, au = oracle.qgemv(u["packed"], u["scales"], u["biases"], x, threads=ORACLE_THREADS)
    assert_within(qg.to_numpy(h).astype(np.float64), oracle.swiglu(gr, ur),
                  swiglu_bound(gr, ur, REL * ag + ABS, REL * au + ABS))


def test_dense_layer_outlier_channels(qg):
    """hidden 5120, FFN 17408 with outlier channels in x: the layer against the fp64 chain."""
    ws = (_w_with_zeros(51, I.TID_GATE, 17408, 5120), _w_with_zeros(51, I.TID_UP, 17408, 5120),
          _w_with_zeros(51, I.TID_DOWN, 5120, 17408))
    x = _x_with_outliers(51, 5120)
    G, U, D = (qg.Int4Weight.from_numpy(w) for w in ws)
    y = qg.to_numpy(qg.dense_layer_int4(G, U, D, qg.to_device(x))).astype(np.float64)
    y_ref, y_bound, _, _ = dense_layer_reference(*ws, x)
    assert_within(y, y_ref, y_bound)


def test_moe_outlier_channels(qg):
    """MoE decode (128 experts, hidden 2048, intermediate 768, top 8) with outlier channels in x."""
    E, hidden, inter, k = 128, 2048, 768, 8
    gate = _w_with_zeros(61, I.TID_GATE, inter, hidden, n_mat=E)
    up = I.int4_weight(61, I.TID_UP, inter, hidden, n_mat=E)
    down = I.int4_weight(61, I.TID_DOWN, hidden, inter, n_mat=E)
    logits = I.f32_normal(61, I.TID_LOGITS, E)
    x = _x_with_outliers(61, hidden)
    r = I.bf16_normal(61, I.TID_RESID, hidden)
    G, U, D = (qg.Int4Weight.from_numpy(d) for d in (gate, up, down))
    y, idx, p = qg.moe_layer_int4(qg.to_device(logits), G, U, D, qg.to_device(x), qg.to_device(r), k=k)
    i_ref, p_ref = oracle.router_topk(logits, k)
    assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist()
    t = lambda d: (d["packed"], d["scales"], d["biases"])  # noqa: E731
    y_ref, a, _ = oracle.moe(t(gate), t(up), t(down), i_ref, p_ref, x, r)
    extra = np.zeros_like(a)
    for s_, e in enumerate(i_ref.tolist()):
        ex = lambda d: tuple(np.ascontiguousarray(v[e]) for v in t(d))  # noqa: E731
        gr, ag = oracle.qgemv(*ex(gate), x)
        ur, au = oracle.qgemv(*ex(up), x)
        _, dab = oracle.qgemv_f64x(*ex(down), swiglu_bound(gr, ur, REL * ag + ABS, REL * au + ABS))
        extra += abs(p_ref[s_]) * dab
    # the down GEMV's bound on the GPU's h plus the gate/up errors carried through SwiGLU
    assert_within(qg.to_numpy(y).astype(np.float64), y_ref, REL * (a + extra) + ABS + extra)


@pytest.mark.parametrize("T", [2, 5, 8])
def test_qgemm_small_t_outlier_channels(qg, T):
    """Small T with outlier channels in the token rows (one row without): T = 2 on the per-token
    GEMV (flagged groups take the second pass), T = 5 and 8 on the tensor cores."""
    d = _w_with_zeros(72, I.TID_W, 1000, 4096)
    X = np.stack([_x_with_outliers(72 + t, 4096) for t in range(T)])
    X[1 % T] = I.bf16_normal(73, I.TID_X, 4096)  # one token without outliers
    Y = qg.to_numpy(qg.qgemm_int4(qg.Int4Weight.from_numpy(d), qg.to_device(X))).astype(np.float64)
    Y_ref, A = oracle.qgemm(d["packed"], d["scales"], d["biases"], X, threads=ORACLE_THREADS)
    assert_within_bound(Y, Y_ref, A)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("T", [32, 40])
def test_qgemm_tensor_core_outlier_channels(qg, T):
    """The tensor-core GEMM with outlier channels in every token row (each row scaled by its own
    largest magnitude, so the N(0,1) entries keep fp16's full precision)."""
    d = _w_with_zeros(71, I.TID_W, 1000, 4096)
    X = np.stack([_x_with_outliers(71 + t, 4096) for t in range(T)])
    Y = qg.to_numpy(qg.qgemm_int4(qg.Int4Weight.from_numpy(d), qg.to_device(X))).astype(np.float64)
    Y_ref, A = oracle.qgemm(d["packed"], d["scales"], d["biases"], X, threads=ORACLE_THREADS)
    assert_within_bound(Y, Y_ref, A)


def test_q2_outlier_channels(qg):
    """The 2-bit GEMV with outlier channels in x."""
    out, in_dim = 1000, 4096
    d = I.int2_weight(81, I.TID_W, out, in_dim)
    x = _x_with_outliers(81, in_dim)
    W = qg.Int4Weight(qg.to_device(d["packed"]), qg.to_device(d["scales"]), qg.to_device(d["biases"]), out, in_dim,
                      bits=2)
    y = qg.to_numpy(qg.qgemv_q2(W, qg.to_device(x))).astype(np.float64)
    y_ref, a = oracle.qgemv2(d["packed"], d["scales"], d["biases"], x, threads=ORACLE_THREADS)
    assert_within_bound(y, y_ref, a)

"""Pins for the fp64 oracle: values the pages print, closed forms, invariants and exact-rational
brute force.  Each check is built so that a plausible slip in the oracle (a dropped bias term, a
wrong group or nibble index, a transposed operand, a missing renormalisation, a wrong SiLU sign,
a dropped residual) fails at least one of them.  CPU only."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from moe_int4_affine_gb300 import inputs as I

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    d = {}
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            d[k] = v
    return d


# ---------------------------------------------------------------- bf16 decode
def _bf16_fraction(bits: int) -> Fraction:
    """bf16 value from its fields (sign, 8-bit exponent, 7-bit fraction), as an exact rational."""
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    assert e != 0xFF
    if e == 0:
        return sign * Fraction(f, 128) * Fraction(2) ** (-126)
    return sign * (1 + Fraction(f, 128)) * Fraction(2) ** (e - 127)


@pytest.mark.parametrize("bits,val", [(0x3F80, 1.0), (0xC000, -2.0), (0x3F81, 1 + 2 ** -7), (0x0000, 0.0),
                                      (0x8000, -0.0), (0x0001, 2.0 ** -133), (0x7F7F, (2 - 2 ** -7) * 2.0 ** 127),
                                      (0x3D80, 0.0625), (0xBE80, -0.25)])
def test_bf16_decode_known_values(bits, val):
    assert oracle.bf16_to_f64(bits) == val
    assert float(_bf16_fraction(bits)) == val


def test_bf16_decode_all_finite_patterns_match_fields():
    for bits in list(range(0, 0x7F80, 97)) + list(range(0x8000, 0xFF80, 89)):
        assert oracle.bf16_to_f64(bits) == float(_bf16_fraction(bits)), hex(bits)


# ---------------------------------------------------------------- nibble unpack
def test_unpack_known_words():
    w = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    q = oracle.unpack(w, 16)
    assert q.tolist() == [list(range(16))]


def test_unpack_every_value_every_position():
    for pos in range(8):
        for v in range(16):
            w = np.array([[v << (4 * pos)]], dtype=np.uint32)
            q = oracle.unpack(w, 8)[0]
            exp = [0] * 8
            exp[pos] = v
            assert q.tolist() == exp, (pos, v)


def test_unpack_random_words_vs_base16_digits():
    g = np.random.default_rng(5)
    words = g.integers(0, 2 ** 32, size=(7, 12), dtype=np.uint64).astype(np.uint32)
    q = oracle.unpack(words, 96)
    for r in range(7):
        for w in range(12):
            n = int(words[r, w])
            digits = []
            for _ in range(8):  # little-endian base-16 digits
                n, d = divmod(n, 16)
                digits.append(d)
            assert q[r, 8 * w:8 * w + 8].tolist() == digits


def test_generator_packing_roundtrip_through_oracle_unpack():
    d = I.int4_weight(0, 99, 5, 192, keep_codes=True)
    assert np.array_equal(oracle.unpack(d["packed"], 192), d["codes"])


# ---------------------------------------------------------------- worked example (golden)
def test_qgemv_worked_example():
    g = _read_golden("qgemv_worked_example.txt")
    out, in_dim = int(g["out"][0]), int(g["in"][0])
    packed = np.array([[int(h, 16) for h in g[f"row{r}_words"]] for r in range(out)], dtype=np.uint32)
    scales = np.array([int(h, 16) for h in g["scales"]], dtype=np.uint16).reshape(out, in_dim // 64)
    biases = np.array([int(h, 16) for h in g["biases"]], dtype=np.uint16).reshape(out, in_dim // 64)
    x = np.array([int(g["x_even"][0], 16) if j % 2 == 0 else int(g["x_odd"][0], 16) for j in range(in_dim)],
                 dtype=np.uint16)
    y, a = oracle.qgemv(packed, scales, biases, x)
    assert y.tolist() == [float(v) for v in g["y"]]
    assert a.tolist() == [float(v) for v in g["absref"]]


# ---------------------------------------------------------------- closed forms
def _weight(out=6, in_dim=256, seed=3):
    return I.int4_weight(seed, 1, out, in_dim, keep_codes=True)


def test_all_zero_codes_gives_bias_times_group_sum():
    d = _weight()
    packed = np.zeros_like(d["packed"])
    x = I.bf16_normal(0, 2, 256)
    y, _ = oracle.qgemv(packed, d["scales"], d["biases"], x)
    xs = [_bf16_fraction(int(b)) for b in x]
    for r in range(6):
        exp = sum(_bf16_fraction(int(d["biases"][r, g])) * sum(xs[64 * g:64 * g + 64]) for g in range(4))
        assert y[r] == pytest.approx(float(exp), rel=1e-14, abs=1e-14)


@pytest.mark.parametrize("j", [0, 1, 7, 8, 63, 64, 65, 127, 128, 200, 255])
def test_one_hot_x_selects_dequantised_column(j):
    d = _weight()
    x = np.zeros(256, dtype=np.uint16)
    x[j] = 0x3F80  # 1.0
    y, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    for r in range(6):
        s = _bf16_fraction(int(d["scales"][r, j // 64]))
        b = _bf16_fraction(int(d["biases"][r, j // 64]))
        w = s * int(d["codes"][r, j]) + b
        assert y[r] == float(w)
        assert a[r] == abs(float(w))


def test_transposed_operand_would_be_caught():
    """Non-square shape with distinct rows: y must depend on the row's own codes only."""
    d = _weight(out=3, in_dim=128)
    x = I.bf16_normal(0, 2, 128)
    y, _ = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    y_rows = [oracle.qgemv(d["packed"][r:r + 1], d["scales"][r:r + 1], d["biases"][r:r + 1], x)[0][0] for r in range(3)]
    assert y.tolist() == y_rows


def test_power_of_two_scaling_is_exact():
    d = _weight()
    x = I.bf16_normal(0, 2, 256)
    y, _ = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    # multiply every scale and bias by 4: exponent field + 2 (no overflow for these values)
    s4 = (d["scales"].astype(np.uint32) + (2 << 7)).astype(np.uint16)
    b4 = np.where(d["biases"] & 0x7F80, d["biases"].astype(np.uint32) + (2 << 7), d["biases"]).astype(np.uint16)
    y4, _ = oracle.qgemv(d["packed"], s4, b4, x)
    np.testing.assert_array_equal(y4, 4.0 * y)


def test_linearity_in_x():
    d = _weight()
    # x1, x2 bf16 with few significant bits so x1 + x2 is exactly representable in bf16
    g = np.random.default_rng(1)
    a1 = g.integers(-8, 9, 256) / 8.0
    a2 = g.integers(-8, 9, 256) / 4.0
    x1, x2, x12 = I.f64_to_bf16_bits(a1), I.f64_to_bf16_bits(a2), I.f64_to_bf16_bits(a1 + a2)
    y1, _ = oracle.qgemv(d["packed"], d["scales"], d["biases"], x1)
    y2, _ = oracle.qgemv(d["packed"], d["scales"], d["biases"], x2)
    y12, _ = oracle.qgemv(d["packed"], d["scales"], d["biases"], x12)
    np.testing.assert_allclose(y12, y1 + y2, rtol=1e-12, atol=1e-12)


def test_f32_input_matches_bf16_input_on_bf16_values():
    d = _weight()
    xb = I.bf16_normal(0, 2, 256)
    y1, a1 = oracle.qgemv(d["packed"], d["scales"], d["biases"], xb)
    y2, a2 = oracle.qgemv(d["packed"], d["scales"], d["biases"], I.bf16_bits_to_f32(xb))
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(a1, a2)


# ---------------------------------------------------------------- exact rational brute force
@pytest.mark.parametrize("out,in_dim", [(1, 64), (3, 64), (2, 128), (3, 128)])
def test_bruteforce_exact_rational(out, in_dim):
    g = np.random.default_rng(out * 1000 + in_dim)
    codes = np.tile(np.arange(16, dtype=np.uint8), out * in_dim // 16).reshape(out, in_dim)
    codes = np.ascontiguousarray(codes[:, g.permutation(in_dim)])  # every code value on every row
    packed = I.pack_codes(codes)
    ng = in_dim // 64
    scales = I.f64_to_bf16_bits(g.uniform(0.005, 0.02, (out, ng)))
    biases = I.f64_to_bf16_bits(g.normal(-0.1, 0.05, (out, ng)))
    x = I.f64_to_bf16_bits(g.standard_normal(in_dim))
    y, a = oracle.qgemv(packed, scales, biases, x)
    for r in range(out):
        acc = Fraction(0)
        aacc = Fraction(0)
        for j in range(in_dim):
            w = _bf16_fraction(int(scales[r, j // 64])) * int(codes[r, j]) + _bf16_fraction(int(biases[r, j // 64]))
            t = w * _bf16_fraction(int(x[j]))
            acc += t
            aacc += abs(t)
        assert abs(Fraction(y[r]) - acc) <= Fraction(1, 10 ** 15) * aacc
        assert abs(Fraction(a[r]) - aacc) <= Fraction(1, 10 ** 15) * aacc


def test_row_range_matches_full():
    d = _weight(out=9)
    x = I.bf16_normal(0, 2, 256)
    y, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    y2, a2 = oracle.qgemv(d["packed"], d["scales"], d["biases"], x, rows=(3, 7))
    np.testing.assert_array_equal(y[3:7], y2)
    y3, _ = oracle.qgemv(d["packed"], d["scales"], d["biases"], x, threads=3)
    np.testing.assert_array_equal(y, y3)


# ---------------------------------------------------------------- SwiGLU
def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle.silu(-40.0)) < 1e-15
    assert oracle.silu(math.log(3.0)) == pytest.approx(math.log(3.0) * 0.75, rel=1e-15)  # sigma(ln 3) = 3/4
    assert oracle.silu(-math.log(3.0)) == pytest.approx(-math.log(3.0) * 0.25, rel=1e-15)
    h = oracle.swiglu(np.array([math.log(3.0), 0.0, -math.log(3.0)]), np.array([2.0, 5.0, -4.0]))
    np.testing.assert_allclose(h, [1.5 * math.log(3.0), 0.0, math.log(3.0)], rtol=1e-15)


# ---------------------------------------------------------------- router
def test_router_pages_example():
    g = _read_golden("router_topk_pages_example.txt")
    logits = np.array([float(v) for v in g["logits"]], dtype=np.float32)
    idx, p = oracle.router_topk(logits, int(g["k"][0]))
    assert idx.tolist() == [int(v) for v in g["idx"]]
    np.testing.assert_allclose(p, [float(v) for v in g["p"]], rtol=1e-15)
    assert p.sum() == pytest.approx(1.0, rel=1e-15)
    assert p[0] > p[1]


def test_router_tie_takes_lower_index():
    logits = np.array([0.5, 2.0, -1.0, 2.0, 2.0, 0.0], dtype=np.float32)
    idx, p = oracle.router_topk(logits, 3)
    assert idx.tolist() == [1, 3, 4]
    np.testing.assert_allclose(p, [1 / 3] * 3, rtol=1e-15)
    idx, _ = oracle.router_topk(logits, 4)
    assert idx.tolist() == [1, 3, 4, 0]


def test_router_full_softmax_variant():
    logits = np.array([1, 5, 3, 4], dtype=np.float32)
    idx, p = oracle.router_topk(logits, 2, renorm=False)
    z = sum(math.exp(v) for v in [1, 5, 3, 4])
    assert idx.tolist() == [1, 3]
    np.testing.assert_allclose(p, [math.exp(5) / z, math.exp(4) / z], rtol=1e-15)


def test_router_k8_of_128_matches_sort():
    logits = I.f32_normal(0, I.TID_LOGITS, 128)
    idx, p = oracle.router_topk(logits, 8)
    order = sorted(range(128), key=lambda e: (-float(logits[e]), e))[:8]
    assert idx.tolist() == order
    assert p.sum() == pytest.approx(1.0, rel=1e-14)
    assert np.all(np.diff(p) <= 0)


# ---------------------------------------------------------------- chain8 + residual
def test_chain_equal_values_and_weights_summing_to_one():
    v1 = I.f32_normal(0, 1, 64)
    v = np.tile(v1, (8, 1))
    p = np.array([0.5, 0.25, 0.125, 0.0625, 0.03125, 0.015625, 0.0078125, 0.0078125])
    r = I.bf16_normal(0, 2, 64)
    y, _ = oracle.chain_residual(p, v, r)
    np.testing.assert_array_equal(y, I.bf16_bits_to_f32(r).astype(np.float64) + v1.astype(np.float64))


@pytest.mark.parametrize("k", range(8))
def test_chain_one_hot_weight_selects_slot(k):
    v = I.f32_normal(0, 1, (8, 64))
    p = np.zeros(8)
    p[k] = 1.0
    r = I.bf16_normal(0, 2, 64)
    y, a = oracle.chain_residual(p, v, r)
    rr = I.bf16_bits_to_f32(r).astype(np.float64)
    np.testing.assert_array_equal(y, rr + v[k].astype(np.float64))
    np.testing.assert_array_equal(a, np.abs(rr) + np.abs(v[k].astype(np.float64)))


# ---------------------------------------------------------------- MoE
def _moe_weights(E=6, hidden=128, inter=64):
    gate = I.int4_weight(0, I.TID_GATE, inter, hidden, n_mat=E)
    up = I.int4_weight(0, I.TID_UP, inter, hidden, n_mat=E)
    down = I.int4_weight(0, I.TID_DOWN, hidden, inter, n_mat=E)
    t = lambda d: (d["packed"], d["scales"], d["biases"])
    return t(gate), t(up), t(down)


def _expert_by_slab(gate, up, down, e, x):
    """The expert computed from slices of the stacked tensors (numpy indexing, not the oracle's
    pointer arithmetic)."""
    g, _ = oracle.qgemv(gate[0][e], gate[1][e], gate[2][e], x)
    u, _ = oracle.qgemv(up[0][e], up[1][e], up[2][e], x)
    h = np.array([gi / (1 + math.exp(-gi)) * ui for gi, ui in zip(g, u)])
    d, _ = oracle.qgemv_f64x(down[0][e], down[1][e], down[2][e], h)
    return d


@pytest.mark.parametrize("e", [0, 3, 5])
def test_moe_one_hot_router_reduces_to_single_expert(e):
    gate, up, down = _moe_weights()
    x = I.bf16_normal(0, 2, 128)
    r = I.bf16_normal(0, 6, 128)
    idx = np.array([e, 1, 2, 3, 4, 0, 1, 2], dtype=np.uint32)
    p = np.array([1.0, 0, 0, 0, 0, 0, 0, 0])
    y, _, flags = oracle.moe(gate, up, down, idx, p, x, r)
    assert flags == 0
    exp = I.bf16_bits_to_f32(r).astype(np.float64) + _expert_by_slab(gate, up, down, e, x)
    np.testing.assert_allclose(y, exp, rtol=1e-13, atol=1e-13)


def test_moe_weighted_sum_of_experts():
    gate, up, down = _moe_weights()
    x = I.bf16_normal(0, 2, 128)
    r = I.bf16_normal(0, 6, 128)
    idx = np.array([5, 2, 0, 1, 3, 4, 2, 5], dtype=np.uint32)
    p = np.array([0.3, 0.2, 0.1, 0.1, 0.1, 0.1, 0.05, 0.05])
    y, a, flags = oracle.moe(gate, up, down, idx, p, x, r)
    exp = I.bf16_bits_to_f32(r).astype(np.float64)
    for k in range(8):
        exp = exp + p[k] * _expert_by_slab(gate, up, down, int(idx[k]), x)
    np.testing.assert_allclose(y, exp, rtol=1e-12, atol=1e-12)
    assert np.all(a >= np.abs(y) - 1e-12)


def test_moe_out_of_range_index_is_skipped_and_flagged():
    gate, up, down = _moe_weights()
    x = I.bf16_normal(0, 2, 128)
    r = I.bf16_normal(0, 6, 128)
    idx = np.array([1, 99, 2, 3, 4, 0, 1, 2], dtype=np.uint32)
    p = np.full(8, 0.125)
    y, _, flags = oracle.moe(gate, up, down, idx, p, x, r)
    assert flags == 1 << 1
    idx2 = idx.copy()
    idx2[1] = 0
    p2 = p.copy()
    p2[1] = 0.0
    y2, _, _ = oracle.moe(gate, up, down, idx2, p2, x, r)
    np.testing.assert_array_equal(y, y2)


# ---------------------------------------------------------------- GEMM
def test_qgemm_rows_equal_qgemv_rows():
    d = _weight(out=5)
    X = I.bf16_normal(0, 2, (3, 256))
    Y, A = oracle.qgemm(d["packed"], d["scales"], d["biases"], X)
    for t in range(3):
        y, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], X[t])
        np.testing.assert_array_equal(Y[t], y)
        np.testing.assert_array_equal(A[t], a)
    Y2, _ = oracle.qgemm(d["packed"], d["scales"], d["biases"], X, rows=(1, 4))
    np.testing.assert_array_equal(Y2, Y[:, 1:4])


def test_qgemm_zero_padding_rows_do_not_change_real_rows():
    d = _weight(out=4)
    X = I.bf16_normal(0, 2, (3, 256))
    Xp = np.zeros((32, 256), dtype=np.uint16)
    Xp[:3] = X
    Y, _ = oracle.qgemm(d["packed"], d["scales"], d["biases"], X)
    Yp, _ = oracle.qgemm(d["packed"], d["scales"], d["biases"], Xp)
    np.testing.assert_array_equal(Yp[:3], Y)
    # padded rows see x = 0, so every term is w*0 and the sum is exactly 0
    np.testing.assert_array_equal(Yp[3:], 0.0)


# ---------------------------------------------------------------- generator sanity (data recipe)
def test_generator_distribution_recipe():
    d = I.int4_weight(0, 1, 256, 1024, keep_codes=True)
    s = I.bf16_bits_to_f32(d["scales"]).astype(np.float64)
    b = I.bf16_bits_to_f32(d["biases"]).astype(np.float64)
    assert s.min() >= 0.005 * (1 - 2 ** -8) and s.max() <= 0.02 * (1 + 2 ** -8)
    assert abs(np.mean(b + 8 * s)) < 2e-4 and 0.5e-3 < np.std(b + 8 * s) < 1.5e-3
    counts = np.bincount(d["codes"].ravel(), minlength=16)
    assert counts.min() > 0.9 * counts.mean()
    x = I.bf16_bits_to_f32(I.bf16_normal(0, 2, 100000)).astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    # reproducible
    d2 = I.int4_weight(0, 1, 256, 1024)
    assert np.array_equal(d["packed"], d2["packed"]) and np.array_equal(d["biases"], d2["biases"])


# ---------------------------------------------------------------- RMSNorm (norm-fused GEMV prologue)
def _bf16_bits(v: float) -> int:
    """bf16 bits of a value exactly representable in bf16."""
    b = np.array([v], dtype=np.float32).view(np.uint32)[0]
    assert b & 0xFFFF == 0, v
    return int(b >> 16)


def test_rmsnorm_worked_example():
    """x = (3, 4), gamma = (1, 2), eps = 0: mean square 12.5, so out = (3, 8) / sqrt(12.5)."""
    out = oracle.rmsnorm(np.array([3.0, 4.0], np.float32), np.array([0x3F80, 0x4000], np.uint16), 0.0)
    assert out[0] == pytest.approx(3 / math.sqrt(12.5), rel=1e-15)
    assert out[1] == pytest.approx(8 / math.sqrt(12.5), rel=1e-15)


@pytest.mark.parametrize("n,j,a", [(64, 0, 2.5), (5120, 4097, -0.75), (17408, 17407, 1e-3)])
def test_rmsnorm_one_hot_closed_form(n, j, a):
    """x = a e_j, gamma = 1, eps = 0: mean square a^2 / n, so out = sqrt(n) sign(a) e_j (a sum in
    place of the mean, or a missing root, fails this)."""
    x = np.zeros(n, np.float32)
    x[j] = a
    out = oracle.rmsnorm(x, np.full(n, 0x3F80, np.uint16), 0.0)
    want = np.zeros(n)
    want[j] = math.copysign(math.sqrt(n), a)
    np.testing.assert_allclose(out, want, rtol=1e-14, atol=0)


def test_rmsnorm_constant_vector_and_gamma():
    """x = c (every element), eps = 0: out = sign(c) gamma, up to the rounding of the fp64 sum of
    n squares (relative error below n 2^-53)."""
    n = 1000
    g = I.bf16_normal(3, I.TID_X, n)
    out = oracle.rmsnorm(np.full(n, -0.3, np.float32), g, 0.0)
    np.testing.assert_allclose(out, -oracle_values(g), rtol=n * 2.0 ** -53)


def oracle_values(bits):
    return np.array([oracle.bf16_to_f64(int(b)) for b in bits])


def test_rmsnorm_scale_invariance_and_epsilon():
    """eps = 0: rmsnorm(alpha x) = rmsnorm(x) for alpha > 0.  eps much larger than the mean
    square: out -> x gamma / sqrt(eps) (eps outside the root, or added to the sum instead of the
    mean, fails this)."""
    n = 2048
    x = I.bf16_normal(4, I.TID_X, n)
    g = I.bf16_normal(5, I.TID_X, n)
    xf = oracle_values(x).astype(np.float32)
    a = oracle.rmsnorm(xf, g, 0.0)
    b = oracle.rmsnorm((xf * np.float32(8.0)).astype(np.float32), g, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-14)
    small = (xf * np.float32(2.0 ** -20)).astype(np.float32)
    eps = 1e4
    c = oracle.rmsnorm(small, g, eps)
    want = small.astype(np.float64) * oracle_values(g) / math.sqrt(eps)
    np.testing.assert_allclose(c, want, rtol=1e-12)
    # the mean of squares, not the sum: with eps = mean square, out = x gamma / sqrt(2 ms)
    ms = float(np.mean(xf.astype(np.float64) ** 2))
    d = oracle.rmsnorm(xf, g, ms)
    np.testing.assert_allclose(d, xf * oracle_values(g) / math.sqrt(2 * ms), rtol=1e-12)


def test_rmsnorm_bf16_and_f32_inputs_agree():
    x = I.bf16_normal(6, I.TID_X, 576)
    g = I.bf16_normal(7, I.TID_X, 576)
    np.testing.assert_array_equal(oracle.rmsnorm(x, g, 1e-6), oracle.rmsnorm(oracle_values(x).astype(np.float32), g, 1e-6))


def test_rmsnorm_qgemv_one_hot_selects_scaled_column():
    """x = a e_j, gamma = g, eps = 0: y = sqrt(n) sign(a) g_j W[:, j], with W[:, j] dequantised
    from the unpacked code and its group's scale and bias."""
    out, n, j = 96, 1024, 777
    d = I.int4_weight(8, I.TID_W, out, n)
    gamma = I.bf16_normal(8, I.TID_X, n)
    x = np.zeros(n, np.float32)
    x[j] = -1.5
    y, _ = oracle.rmsnorm_qgemv(d["packed"], d["scales"], d["biases"], x, gamma, 0.0)
    q = oracle.unpack(d["packed"], n)[:, j].astype(np.float64)
    s = oracle_values(d["scales"].reshape(out, n // 64)[:, j // 64])
    b = oracle_values(d["biases"].reshape(out, n // 64)[:, j // 64])
    want = -math.sqrt(n) * oracle.bf16_to_f64(int(gamma[j])) * (s * q + b)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------- sigmoid-gated scalar FMA (shared expert)
def test_sigmoid_closed_forms():
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.sigmoid(math.log(3.0)) == pytest.approx(0.75, rel=1e-15)
    assert oracle.sigmoid(-math.log(3.0)) == pytest.approx(0.25, rel=1e-15)
    assert oracle.sigmoid(40.0) == pytest.approx(1.0, abs=1e-17)
    assert 0.0 < oracle.sigmoid(-40.0) < 1e-17


def test_sigmoid_scalar_fma_closed_forms():
    """gate = ln 3 -> sigmoid 3/4; gate = 0 -> 1/2; gate = -40 -> base + residual only; and the
    residual (bf16) is added once, with the variant without it matching base + s v."""
    n = 300
    v = I.f32_normal(9, I.TID_X, n)
    base = I.f32_normal(10, I.TID_X, n)
    r = I.bf16_normal(11, I.TID_RESID, n)
    rv = oracle_values(r)
    out, a = oracle.sigmoid_scalar_fma(math.log(3.0), v, base, r)
    np.testing.assert_allclose(out, base + 0.75 * v.astype(np.float64) + rv, rtol=1e-14, atol=1e-15)
    b64, v64 = base.astype(np.float64), v.astype(np.float64)
    np.testing.assert_allclose(a, np.abs(b64) + 0.75 * np.abs(v64) + np.abs(rv), rtol=1e-14)
    out0, _ = oracle.sigmoid_scalar_fma(0.0, v, base)
    np.testing.assert_allclose(out0, base + 0.5 * v.astype(np.float64), rtol=1e-15, atol=1e-16)
    outm, _ = oracle.sigmoid_scalar_fma(-40.0, v, base, r)
    np.testing.assert_allclose(outm, base + rv, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- affine quantizer (encode), next row N3
def _grid_group(rng, bits, s_bits=0x3C50, k=-20):
    """A group on an exact grid: s bf16 (here 0.0126953125), b = k s, w_j = b + q_j s with q_j
    random in [0, 2^bits - 1] and both ends present; every value exact in binary32."""
    qmax = (1 << bits) - 1
    q = rng.integers(0, qmax + 1, 64)
    q[rng.integers(0, 64)] = 0
    q[rng.integers(0, 64)] = qmax
    if q.min() != 0:
        q[np.argmin(q)] = 0
    s = oracle.bf16_to_f64(s_bits)
    w = ((k + q) * s).astype(np.float32)
    return q, s, k * s, w


@pytest.mark.parametrize("bits", [4, 2])
def test_quantize_exact_grid_round_trip(bits):
    """Values on an exact grid b + q s (both ends present): scale s, bias b and every code q come
    back exactly; the packing order is low bits first."""
    rng = np.random.default_rng(bits)
    q, s, b, w = _grid_group(rng, bits)
    packed, sc, bi = oracle.quantize(w.reshape(1, 64), bits)
    assert oracle.bf16_to_f64(int(sc[0, 0])) == s and oracle.bf16_to_f64(int(bi[0, 0])) == b
    per = 32 // bits
    got = [(int(packed[0, j // per]) >> (bits * (j % per))) & ((1 << bits) - 1) for j in range(64)]
    assert got == q.tolist()


def test_quantize_constant_group():
    w = np.full((2, 128), 0.3, np.float32)
    packed, sc, bi = oracle.quantize(w)
    assert np.all(packed == 0) and np.all(sc == 0)
    assert np.all(bi == oracle.bf16_round(np.float32(0.3)))


def test_quantize_zero_groups_store_positive_zero():
    """Groups of zeros of both signs, whichever sign comes first, store scale +0 and bias +0 and
    codes 0 (the range of a set of zeros is zero, not -0)."""
    w = np.zeros((3, 64), np.float32)
    w[0, 0::2] = -0.0
    w[1, :] = -0.0
    w[2, 1::2] = -0.0
    for bits in (4, 2):
        packed, sc, bi = oracle.quantize(w, bits)
        assert np.all(sc == 0) and np.all(bi == 0) and np.all(packed == 0)


def test_quantize_ties_round_to_even():
    """w = (k + 1/2) s exactly (s = 2^-4, b = 0): the code is the even one of k and k + 1; one ulp
    above the tie rounds up, one ulp below rounds down."""
    k = np.arange(15)
    h = ((k + 0.5) / 16).astype(np.float32)
    w = np.full((3, 64), 0.5, np.float32)
    for r, vals in enumerate((h, np.nextafter(h, np.float32(1)), np.nextafter(h, np.float32(0)))):
        w[r, 0], w[r, 1] = 0.0, 15 / 16
        w[r, 2:17] = vals
    packed, sc, bi = oracle.quantize(w, 4)
    assert np.all(sc == 0x3D80) and np.all(bi == 0)  # 2^-4 and 0
    codes = (packed[:, :, None] >> (4 * np.arange(8))) & 0xF
    codes = codes.reshape(3, 64)[:, 2:17]
    assert codes[0].tolist() == [int(c + (c % 2)) for c in k]   # ties: the even neighbour
    assert codes[1].tolist() == (k + 1).tolist()
    assert codes[2].tolist() == k.tolist()


def test_quantize_codes_come_from_bf16_scale_and_bias():
    """lo = 0, hi = 1: with the binary32 scale 1/15, w = 0.968 sits at 14.52 (code 15); with the
    bf16 scale 0.06689453125 at 14.47 (code 14) -- the codes are derived from the rounded scale,
    as the pages require."""
    w = np.zeros(64, np.float32)
    w[1] = 1.0
    w[2] = 0.968
    packed, sc, bi = oracle.quantize(w.reshape(1, 64))
    s = oracle.bf16_to_f64(int(sc[0, 0]))
    assert s == 0.06689453125 and bi[0, 0] == 0
    q2 = (int(packed[0, 0]) >> 8) & 0xF
    assert q2 == 14
    assert np.rint(np.float32(0.968) / (np.float32(1.0) / np.float32(15))) == 15  # unrounded scale


@pytest.mark.parametrize("bits", [4, 2])
def test_quantize_nearest_grid_point_and_error_bound(bits):
    """Random groups: every code is the nearest grid point b + q s in exact arithmetic (clamped to
    [0, 2^bits - 1]), except within 1e-5 of a tie, where binary32 decides; and the dequantised value
    is within s/2 plus the bf16 rounding of scale and bias of the input."""
    rng = np.random.default_rng(10 + bits)
    qmax = (1 << bits) - 1
    w = rng.normal(0, 0.05, (8, 256)).astype(np.float32)
    packed, sc, bi = oracle.quantize(w, bits)
    per = 32 // bits
    for r in range(8):
        for g in range(4):
            s = oracle.bf16_to_f64(int(sc[r, g]))
            b = oracle.bf16_to_f64(int(bi[r, g]))
            grp = w[r, 64 * g:64 * g + 64].astype(np.float64)
            lo, hi = grp.min(), grp.max()
            assert abs(b - lo) <= abs(lo) * 2.0 ** -8 and s > 0
            for j in range(64):
                col = 64 * g + j
                q = (int(packed[r, col // per]) >> (bits * (col % per))) & qmax
                t = (grp[j] - b) / s
                frac = t - math.floor(t)
                if abs(frac - 0.5) > 1e-5:
                    assert q == min(max(int(math.floor(t + 0.5)), 0), qmax), (r, g, j, t, q)
                err = abs(grp[j] - (b + q * s))
                assert err <= s / 2 + abs(b - lo) + qmax * abs(s - (hi - lo) / qmax) + 1e-12


def test_quantize_bf16_and_f32_inputs_agree():
    x = I.bf16_normal(12, I.TID_X, (4, 192))
    a = oracle.quantize(x)
    b = oracle.quantize(np.array([[oracle.bf16_to_f64(int(v)) for v in row] for row in x], np.float32))
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


# ---------------------------------------------------------------- 2-bit GEMV (Q2_64A), next row N4
def test_code2_known_words():
    w = np.array([[0xE4E4E4E4, 0x00000003]], np.uint32)  # 0xE4 = codes 0,1,2,3 (low first)
    assert [oracle.code2(w, 32, 0, j) for j in range(16)] == [0, 1, 2, 3] * 4
    assert [oracle.code2(w, 32, 0, j) for j in range(16, 32)] == [3] + [0] * 15


def _q2_weight(seed, out, in_dim):
    rng = np.random.default_rng(seed)
    packed = rng.integers(0, 2 ** 32, (out, in_dim // 16), dtype=np.uint64).astype(np.uint32)
    s = np.array([oracle.bf16_round(v) for v in rng.uniform(0.005, 0.02, out * in_dim // 64)], np.uint16)
    b = np.array([oracle.bf16_round(v) for v in rng.normal(-0.02, 0.01, out * in_dim // 64)], np.uint16)
    return packed, s.reshape(out, -1), b.reshape(out, -1)


def test_qgemv2_all_zero_codes_and_one_hot():
    """Codes all 0: y = sum_g b_g * sum_{j in g} x_j; one-hot x: y = s q + b of that column."""
    out, n = 9, 192
    packed, s, b = _q2_weight(1, out, n)
    x = I.bf16_normal(1, I.TID_X, n)
    xv = oracle_values(x)
    y0, _ = oracle.qgemv2(np.zeros_like(packed), s, b, x)
    want = [sum(oracle.bf16_to_f64(int(b[r, g])) * xv[64 * g:64 * g + 64].sum() for g in range(3)) for r in range(out)]
    np.testing.assert_allclose(y0, want, rtol=1e-12)
    for j in (0, 17, 100, 191):
        e = np.zeros(n, np.float32)
        e[j] = 1.0
        y, _ = oracle.qgemv2(packed, s, b, e)
        col = [oracle.bf16_to_f64(int(s[r, j // 64])) * oracle.code2(packed, n, r, j) + oracle.bf16_to_f64(int(b[r, j // 64]))
               for r in range(out)]
        np.testing.assert_array_equal(y, col)


def test_qgemv2_bruteforce_exact_rational():
    out, n = 3, 128
    packed, s, b = _q2_weight(2, out, n)
    x = I.bf16_normal(2, I.TID_X, n)
    y, _ = oracle.qgemv2(packed, s, b, x)
    for r in range(out):
        exact = Fraction(0)
        for j in range(n):
            word = int(packed[r, j // 16])
            q = (word >> (2 * (j % 16))) & 3
            exact += (_bf16_fraction(int(s[r, j // 64])) * q + _bf16_fraction(int(b[r, j // 64]))) * _bf16_fraction(int(x[j]))
        assert abs(Fraction(y[r]) - exact) <= abs(exact) * Fraction(1, 2 ** 40) + Fraction(1, 2 ** 60)


def test_qgemv2_of_the_2bit_encoding():
    """The encoder's 2-bit output read back by the 2-bit GEMV: with one-hot x every column is its
    dequantised weight b + q s, within s/2 + bf16 effects of the original weight."""
    rng = np.random.default_rng(3)
    w = rng.normal(0, 0.03, (4, 128)).astype(np.float32)
    packed, s, b = oracle.quantize(w, 2)
    for j in (0, 63, 64, 127):
        e = np.zeros(128, np.float32)
        e[j] = 1.0
        y, _ = oracle.qgemv2(packed, s, b, e)
        for r in range(4):
            sv = oracle.bf16_to_f64(int(s[r, j // 64]))
            assert abs(y[r] - w[r, j]) <= sv / 2 + abs(w[r, 64 * (j // 64):64 * (j // 64) + 64]).max() * 2.0 ** -7


def _repack_2bit_as_4bit(packed2, in_dim):
    """The 2-bit codes of a weight as 4-bit codes (values 0..3), eight per u32, low first."""
    lead = packed2.shape[:-1]
    words = packed2.reshape(-1, in_dim // 16).astype(np.uint64)
    codes = (words[:, :, None] >> (2 * np.arange(16, dtype=np.uint64))) & 3
    codes = codes.reshape(words.shape[0], in_dim // 8, 8)
    out = (codes << (4 * np.arange(8, dtype=np.uint64))).sum(axis=2).astype(np.uint32)
    return out.reshape(lead + (in_dim // 8,))


def test_qgemv2_equals_4bit_path_on_repacked_codes():
    """2-bit codes are valid 4-bit codes: the 2-bit GEMV equals the (pinned) 4-bit GEMV of the same
    weights repacked eight per word, bit for bit."""
    d = I.int2_weight(4, I.TID_W, 50, 576)
    x = I.bf16_normal(4, I.TID_X, 576)
    y2, a2 = oracle.qgemv2(d["packed"], d["scales"], d["biases"], x)
    y4, a4 = oracle.qgemv(_repack_2bit_as_4bit(d["packed"], 576), d["scales"], d["biases"], x)
    np.testing.assert_array_equal(y2, y4)
    np.testing.assert_array_equal(a2, a4)


def test_moe2_equals_4bit_moe_on_repacked_codes():
    E, hidden, inter = 6, 256, 192
    g = I.int2_weight(5, I.TID_GATE, inter, hidden, n_mat=E)
    u = I.int2_weight(5, I.TID_UP, inter, hidden, n_mat=E)
    d = I.int2_weight(5, I.TID_DOWN, hidden, inter, n_mat=E)
    idx = np.array([4, 1, 5], np.uint32)
    p = np.array([0.5, 0.3, 0.2])
    x = I.bf16_normal(5, I.TID_X, hidden)
    r = I.bf16_normal(5, I.TID_RESID, hidden)
    t = lambda w: (w["packed"], w["scales"], w["biases"])
    y2, a2, f2 = oracle.moe2(t(g), t(u), t(d), idx, p, x, r)
    rp = lambda w, n: (_repack_2bit_as_4bit(w["packed"], n), w["scales"], w["biases"])
    y4, a4, f4 = oracle.moe(rp(g, hidden), rp(u, hidden), rp(d, inter), idx, p, x, r)
    np.testing.assert_array_equal(y2, y4)
    np.testing.assert_array_equal(a2, a4)
    assert f2 == f4 == 0


# ---------------------------------------------------------------- gated RMSNorm (Mamba2-style, GDN tail)
def _bf(vals):
    """bf16 bits of values exactly representable in bf16."""
    v = np.asarray(vals, dtype=np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def test_gated_rmsnorm_large_gate_is_rmsnorm_times_gate():
    """silu(t) = t exactly in binary64 for t = 64 (1 / (1 + e^-64) rounds to 1): with z = 64 everywhere
    and one head, the gated norm is 64 times the plain RMSNorm, which is pinned on its own."""
    y = I.bf16_normal(21, I.TID_X, 256)
    g = I.bf16_normal(22, I.TID_RESID, 256)
    z = _bf(np.full(256, 64.0))
    out = oracle.gated_rmsnorm(y, z, g, 1e-6, 256)
    np.testing.assert_allclose(out, 64.0 * oracle.rmsnorm(y, g, 1e-6), rtol=1e-15, atol=0)


def test_gated_rmsnorm_zero_gate_and_silu_values():
    """z = 0 gives 0 (silu(0) = 0); z = +-1 gives silu(1) = 1/(1+e^-1) and silu(-1) = -1/(1+e)."""
    y = _bf([1.0, -2.0, 3.0, 0.5])
    g = _bf([1.0, 1.0, 1.0, 1.0])
    r = math.sqrt((1 + 4 + 9 + 0.25) / 4)
    out = oracle.gated_rmsnorm(y, _bf([0.0, 1.0, -1.0, 0.0]), g, 0.0, 4)
    assert out[0] == 0.0 and out[3] == 0.0
    assert abs(out[1] - (1 / (1 + math.exp(-1))) * (-2.0 / r)) < 1e-15
    assert abs(out[2] - (-1 / (1 + math.e)) * (3.0 / r)) < 1e-15


@pytest.mark.parametrize("head_dim", [64, 128])
def test_gated_rmsnorm_heads_are_independent(head_dim):
    """Per head, with gamma = 1 and z = 64: the output over 64 has mean square 1 (eps = 0), and
    scaling one head's y by 8 changes no output anywhere."""
    n = 512
    y = I.f32_normal(23, I.TID_X, n)
    z = np.full(n, 64.0, np.float32)
    g = _bf(np.ones(n))
    out = oracle.gated_rmsnorm(y, z, g, 0.0, head_dim) / 64.0
    ms = (out.reshape(-1, head_dim) ** 2).mean(axis=1)
    np.testing.assert_allclose(ms, 1.0, rtol=1e-13)
    y2 = y.copy()
    y2[head_dim:2 * head_dim] *= np.float32(8.0)
    np.testing.assert_allclose(oracle.gated_rmsnorm(y2, z, g, 0.0, head_dim) / 64.0, out, rtol=1e-14, atol=0)


def test_gated_rmsnorm_rejects_bad_heads():
    y = I.f32_normal(24, I.TID_X, 96)
    with pytest.raises(ValueError):
        oracle.gated_rmsnorm(y, y, _bf(np.ones(96)), 1e-6, 64)

"""GPU parity of quantize_affine_q64a (the affine group-64 encoder, Q4_64A and Q2_64A) against the
oracle's encoder: codes, scales and biases bit-exact (the code decision is made in binary32 on
both sides), including crafted groups (constant, signed zeros, an exact grid, a code that the bf16
scale moves, scales too small or too large for the reciprocal, quotients on and next to
half-integers), and the encoder's output fed to the GEMV."""
import numpy as np
import pytest

import oracle
from conftest import assert_within_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _weights(seed, out, in_dim, kind):
    rng = np.random.default_rng(seed)
    w = rng.normal(0, 0.02, (out, in_dim)).astype(np.float32)
    if out >= 4 and in_dim >= 128:
        w[0, :64] = 0.3                     # constant group
        w[1, :64] = 0.0                     # zeros of both signs
        w[1, 1:64:2] = -0.0
        w[1, 5] = 0.25
        w[2, :64] = 0.0                     # a code moved by the bf16 scale
        w[2, 1] = 1.0
        w[2, 2] = 0.968
        k = np.arange(64) % 16              # an exact grid
        w[3, 64:128] = ((k - 20) * np.float32(0.0126953125)).astype(np.float32)
    if out >= 8 and in_dim >= 128:
        k = np.arange(64)
        w[4, :64] = (k % 5) * np.float32(2.0 ** -130)     # subnormal weights: 1/s overflows binary32
        w[5, 64:128] = (k % 16) * np.float32(2.0 ** 122)  # s = 2^122: beyond the reciprocal's range
        w[6, :64] = (k % 16) * np.float32(2.0 ** -118)    # s = 2^-118: the smallest scales of the fast path
        w[7, :64] = 0.0                                   # zeros, -0 first
        w[7, 0::2] = -0.0
    if out >= 9 and in_dim >= 128:
        # quotients on and next to every half-integer: s = 2^-4, b = 0 for 4 bits
        h = (np.arange(15, dtype=np.float32) + np.float32(0.5)) / np.float32(16)
        t = np.concatenate([[0.0, 15 / 16], h, np.nextafter(h, np.float32(1)), np.nextafter(h, np.float32(0))])
        w[8, :64] = np.float32(0.5)
        w[8, :t.size] = t.astype(np.float32)
    if kind == "bf16":
        bits = (w.view(np.uint32) + 0x7FFF + ((w.view(np.uint32) >> 16) & 1)) >> 16
        return bits.astype(np.uint16)
    return w


def _gpu(qg, w, bits):
    p, s, b = qg.quantize_affine_q64a(qg.to_device(w), bits)
    return qg.to_numpy(p), qg.to_numpy(s), qg.to_numpy(b)


@pytest.mark.parametrize("out,in_dim", [(1, 64), (5, 128), (37, 576), (256, 1024), (300, 5120)])
@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_quantize_bit_exact_vs_oracle(qg, out, in_dim, bits, kind):
    w = _weights(out + in_dim + bits, out, in_dim, kind)
    p, s, b = _gpu(qg, w, bits)
    pr, sr, br = oracle.quantize(w, bits)
    np.testing.assert_array_equal(s, sr)
    np.testing.assert_array_equal(b, br)
    np.testing.assert_array_equal(p.astype(np.uint32), pr)
    assert qg.qg_device_status() == 0


def test_quantize_full_size_every_row(qg):
    """17408 x 5120 bf16 weights (the FFN gate's shape): every code, scale and bias bit for bit."""
    w = _weights(7, 17408, 5120, "bf16")
    p, s, b = _gpu(qg, w, 4)
    pr, sr, br = oracle.quantize(w, 4)
    np.testing.assert_array_equal(s, sr)
    np.testing.assert_array_equal(b, br)
    np.testing.assert_array_equal(p.astype(np.uint32), pr)


def test_quantized_weights_feed_the_gemv(qg):
    """Encode on the GPU, then the GEMV on the encoded weights matches the oracle's GEMV of the
    oracle's encoding of the same weights (the encodings being identical)."""
    out, in_dim = 1000, 2048
    w = _weights(11, out, in_dim, "f32")
    p, s, b = qg.quantize_affine_q64a(qg.to_device(w), 4)
    W = qg.Int4Weight(p, s, b, out, in_dim)
    x = I.bf16_normal(11, I.TID_X, in_dim)
    y = qg.to_numpy(qg.qgemv_int4(W, qg.to_device(x))).astype(np.float64)
    pr, sr, br = oracle.quantize(w, 4)
    y_ref, a = oracle.qgemv(pr, sr, br, x)
    assert_within_bound(y, y_ref, a)

"""Seeded synthetic inputs for the int4 affine decode path.

This module only draws random data and stores it in the library's input formats (u32-packed
nibbles, bf16 bit patterns, fp32).  It holds none of the path's arithmetic: no dequantisation,
no dot products, no routing.  Tests and the benchmark feed the same arrays to the CUDA library
and to the CPU oracle.

Generator: numpy's PCG64 seeded through a SeedSequence of (seed, tensor id), so each tensor is
an independent, reproducible stream.  Distributions (the workloads the pages decode with; all
synthetic, no checkpoint is involved):
  codes    uniform integers 0..15
  scale    uniform [0.005, 0.02] drawn in float64, rounded to bf16 (nearest, ties to even)
  bias     -8 * scale_bf16 + N(0, 1e-3) drawn in float64, rounded to bf16
  x, residual   N(0, 1) rounded to bf16
  router logits N(0, 1) as float32
"""
from __future__ import annotations

import numpy as np

GROUP = 64


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(tensor_id)])))


def f64_to_bf16_bits(a) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even); return the 16-bit patterns.

    Rounds once, from float64, to 8 significant bits.  Valid for finite values in bf16's normal
    range, which covers every distribution drawn here.
    """
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)
    m = np.round(m * 256.0) / 256.0
    r = np.ldexp(m, e)
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact).  A storage conversion for callers that want to
    look at the data; it is not used to compute any result."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Pack uint8 codes [..., in] (values 0..15) into u32 words [..., in/8]: element 8w+i of a row
    goes to bits 4i..4i+3 of word w (low nibble first)."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape[-1] % 8 == 0
    c = codes.reshape(codes.shape[:-1] + (codes.shape[-1] // 8, 8)).astype(np.uint32)
    words = np.zeros(c.shape[:-1], dtype=np.uint32)
    for i in range(8):
        words |= c[..., i] << np.uint32(4 * i)
    return words


def int4_weight(seed: int, tensor_id: int, out: int, in_dim: int, n_mat: int | None = None,
                keep_codes: bool = False) -> dict:
    """A random int4 affine group-64 weight [out][in] (stacked [n_mat][out][in] if n_mat).

    Returns dict(packed=u32 [.., out, in/8], scales=u16 [.., out, in/64], biases=u16 [.., out, in/64],
    codes=u8 [.., out, in] when keep_codes).
    """
    assert in_dim % GROUP == 0
    lead = () if n_mat is None else (n_mat,)
    g = rng(seed, tensor_id)
    codes = g.integers(0, 16, size=lead + (out, in_dim), dtype=np.uint8)
    s64 = g.uniform(0.005, 0.02, size=lead + (out, in_dim // GROUP))
    scales = f64_to_bf16_bits(s64)
    s_b = bf16_bits_to_f32(scales).astype(np.float64)
    biases = f64_to_bf16_bits(-8.0 * s_b + g.normal(0.0, 1e-3, size=s_b.shape))
    d = dict(packed=pack_codes(codes), scales=scales, biases=biases)
    if keep_codes:
        d["codes"] = codes
    return d


def int2_weight(seed: int, tensor_id: int, out: int, in_dim: int, n_mat: int | None = None) -> dict:
    """A random 2-bit affine group-64 weight [out][in] (the Q2_64A layout): codes uniform 0..3
    packed sixteen per u32 (low first), scales U[0.005, 0.02], biases -1.5 s + N(0, 1e-3) (the
    4-bit recipe with the code midpoint 1.5), bf16.  dict(packed=u32 [.., out, in/16], scales,
    biases); stacked [n_mat][out][in] when n_mat is given."""
    assert in_dim % GROUP == 0
    lead = () if n_mat is None else (n_mat,)
    g = rng(seed, tensor_id)
    codes = g.integers(0, 4, size=lead + (out, in_dim), dtype=np.uint32)
    shifts = (2 * np.arange(16, dtype=np.uint32))
    packed = (codes.reshape(lead + (out, in_dim // 16, 16)) << shifts).sum(axis=-1, dtype=np.uint64).astype(np.uint32)
    s64 = g.uniform(0.005, 0.02, size=lead + (out, in_dim // GROUP))
    scales = f64_to_bf16_bits(s64)
    s_b = bf16_bits_to_f32(scales).astype(np.float64)
    biases = f64_to_bf16_bits(-1.5 * s_b + g.normal(0.0, 1e-3, size=s_b.shape))
    return dict(packed=packed, scales=scales, biases=biases)


def bf16_normal(seed: int, tensor_id: int, shape) -> np.ndarray:
    return f64_to_bf16_bits(rng(seed, tensor_id).standard_normal(shape))


def f32_normal(seed: int, tensor_id: int, shape) -> np.ndarray:
    return rng(seed, tensor_id).standard_normal(shape).astype(np.float32)


# Tensor ids used by the configurations (kept in one place so tests and bench agree).
TID_W = 1
TID_X = 2
TID_GATE = 3
TID_UP = 4
TID_DOWN = 5
TID_RESID = 6
TID_LOGITS = 7
TID_MULTI = 10  # + projection index

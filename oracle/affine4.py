"""Affine 4-bit, group-64 weight format (test infrastructure only).

Follows oxinfer (docs.rs crate page), section "MLX checkpoints": each matrix
row stores packed 4-bit values, eight per uint32, plus one bf16 scale and one
bf16 bias per group of 64 consecutive input elements, and the weight is
w = scale * q + bias.  Nibble order (not fixed by the page): nibble k of word
j holds input element 8j + k in bits 4k..4k+3.
"""

from __future__ import annotations

import numpy as np

from .numerics import bf16_bits_to_f64

GROUP = 64


def unpack_nibbles(words) -> np.ndarray:
    """uint32 words [out, in/8] -> integer codes q [out, in] in 0..15 (int64)."""
    w = np.asarray(words).astype(np.uint32)
    out, n8 = w.shape
    q = np.empty((out, n8 * 8), dtype=np.int64)
    for k in range(8):
        q[:, k::8] = (w >> np.uint32(4 * k)) & np.uint32(0xF)
    return q


def dequant_affine4_g64(words, scales_bits, biases_bits) -> np.ndarray:
    """Exact float64 weights scale * q + bias, shape [out, in]."""
    q = unpack_nibbles(words).astype(np.float64)
    s = bf16_bits_to_f64(scales_bits)
    b = bf16_bits_to_f64(biases_bits)
    out, n = q.shape
    assert s.shape == (out, n // GROUP) and b.shape == s.shape
    s_full = np.repeat(s, GROUP, axis=1)
    b_full = np.repeat(b, GROUP, axis=1)
    return s_full * q + b_full


def dequant_affine4_g64_f32(words, scales_bits, biases_bits) -> np.ndarray:
    """The same weights rounded once to float32 (the bit-exact reference for a
    device dequantiser that evaluates scale * q + bias with one rounding)."""
    return dequant_affine4_g64(words, scales_bits, biases_bits).astype(np.float32)

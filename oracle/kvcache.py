"""KV cache storage formats for the oracle (TEST INFRASTRUCTURE ONLY, see the package header).

Two formats hold the post-norm, post-RoPE keys and the values of every cached slot:

  * bf16: [L][2][B][n_kv][max_ctx][d] bit patterns; an appended row is rounded to bf16.
  * affine 8-bit, groups of 64 ("affine8_g64"): codes uint8 [L][2][B][n_kv][max_ctx][d]
    and, per group of 64 consecutive elements of a row, a bf16 scale and bias
    [L][2][B][n_kv][max_ctx][d/64] (params[..., 0] scale, params[..., 1] bias);
    value = scale * code + bias.

Sources: Butter architecture.md, section on the model layer (per-layer cache types:
KVCache, AffineQuantizedKVCache) and its component list (Caches: KVCache,
AffineQuantizedKVCache); oxinfer crate page, "MLX checkpoints" (the affine form
w = scale * q + bias with one bf16 scale and bias per group of 64).

Readings where the pages are silent:
  * 8-bit codes, groups of 64 consecutive elements of one row (one position of one
    head), bf16 scale and bias, like the affine weight format.
  * Min-max quantization, decided in float32: mn, mx = min, max of the group;
    scale = bf16(fl32(fl32(mx - mn) / 255)); bias = bf16(mn) (round to nearest even);
    code = clamp(rint(fl32(fl32(x - bias) / scale)), 0, 255) with rint rounding halves
    to even, and code = 0 when the scale is 0.  The oracle rounds its float64 row to
    float32 first: the quantizer takes its integer decisions in float32.
  * Reading a row: scale * code + bias, exact in float64.
"""

from __future__ import annotations

import numpy as np

from .numerics import bf16_bits_to_f64, f64_to_bf16_bits

GROUP = 64
LEVELS = 255


def quantize_affine8_g64(x) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Quantize rows x [..., d] (d a multiple of 64).  Returns (codes uint8 [..., d],
    scale bits uint16 [..., d/64], bias bits uint16 [..., d/64])."""
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] % GROUP == 0
    g = x.reshape(*x.shape[:-1], x.shape[-1] // GROUP, GROUP)
    mn = g.min(axis=-1)
    mx = g.max(axis=-1)
    span = np.subtract(mx, mn, dtype=np.float32)
    scale32 = np.divide(span, np.float32(LEVELS), dtype=np.float32)
    scale_bits = f64_to_bf16_bits(scale32.astype(np.float64))
    bias_bits = f64_to_bf16_bits(mn.astype(np.float64))
    s = bf16_bits_to_f64(scale_bits).astype(np.float32)[..., None]
    b = bf16_bits_to_f64(bias_bits).astype(np.float32)[..., None]
    t = np.divide(np.subtract(g, b, dtype=np.float32), np.where(s == 0, np.float32(1), s), dtype=np.float32)
    codes = np.where(s == 0, 0.0, np.clip(np.rint(t), 0, LEVELS)).astype(np.uint8)
    return codes.reshape(x.shape), scale_bits, bias_bits


def dequant_affine8_g64(codes, scale_bits, bias_bits) -> np.ndarray:
    """scale * code + bias per group of 64, exact in float64."""
    c = np.asarray(codes).astype(np.float64)
    g = c.reshape(*c.shape[:-1], c.shape[-1] // GROUP, GROUP)
    s = bf16_bits_to_f64(scale_bits)[..., None]
    b = bf16_bits_to_f64(bias_bits)[..., None]
    return (s * g + b).reshape(c.shape)


class Affine8Cache:
    """Affine 8-bit cache: codes uint8 [L][2][B][n_kv][max_ctx][d], params uint16
    (bf16 bits) [L][2][B][n_kv][max_ctx][d/64][2] = (scale, bias)."""

    def __init__(self, codes: np.ndarray, params: np.ndarray):
        assert codes.dtype == np.uint8 and codes.ndim == 6
        assert params.dtype == np.uint16 and params.shape == codes.shape[:5] + (codes.shape[5] // GROUP, 2)
        self.codes = codes
        self.params = params

    @property
    def shape(self):
        return self.codes.shape

    def copy(self) -> "Affine8Cache":
        return Affine8Cache(self.codes.copy(), self.params.copy())

    def store(self, l: int, plane: int, b: int, P: int, rows: np.ndarray) -> None:
        """Quantize rows [n_kv, d] (float64 values, taken to float32) into slot P."""
        c, s, bb = quantize_affine8_g64(rows)
        self.codes[l, plane, b, :, P, :] = c
        self.params[l, plane, b, :, P, :, 0] = s
        self.params[l, plane, b, :, P, :, 1] = bb

    def read(self, l: int, plane: int, b: int, T: int) -> np.ndarray:
        """float64 [n_kv, T, d] values of slots 0..T-1."""
        p = self.params[l, plane, b, :, :T]
        return dequant_affine8_g64(self.codes[l, plane, b, :, :T], p[..., 0], p[..., 1])


def kv_store(kv, l: int, plane: int, b: int, P: int, rows: np.ndarray) -> None:
    """Write one new row per KV head at slot P in the cache's own format (bf16: round
    to nearest even; affine 8-bit: quantize)."""
    if isinstance(kv, Affine8Cache):
        kv.store(l, plane, b, P, rows)
    else:
        kv[l, plane, b, :, P, :] = f64_to_bf16_bits(rows)


def kv_read(kv, l: int, plane: int, b: int, T: int) -> np.ndarray:
    """float64 [n_kv, T, d]: the values of slots 0..T-1 as the cache holds them."""
    if isinstance(kv, Affine8Cache):
        return kv.read(l, plane, b, T)
    return bf16_bits_to_f64(kv[l, plane, b, :, :T, :])

// Affine 4-bit group-64 decoding shared by the GEMV kernels and the dequant test hook.
//
// Format (oxinfer crate page, "MLX checkpoints"): eight 4-bit codes q per uint32,
// one bf16 scale s and bias b per group of 64 inputs, w = s*q + b.  Code k of a
// word sits in bits 4k..4k+3.  The handle stores (s, b) of a (row, group) as one
// uint32: s in the low 16 bits, b in the high 16 bits.
#pragma once
#include <cstdint>

namespace dec {

// 128 + q as a float, built without a conversion instruction: the code is masked
// into mantissa bits 16..19 of 0x43000000 (= 128.0f, whose mantissa unit at bit 16
// is 1.0), so the result is exactly 128 + q.
template <int K>
__device__ __forceinline__ float q4_code_plus128(uint32_t word) {
  uint32_t v;
  if constexpr (K < 4) {
    v = word << (16 - 4 * K);
  } else if constexpr (K == 4) {
    v = word;
  } else {
    v = word >> (4 * K - 16);
  }
  return __uint_as_float((v & 0x000f0000u) | 0x43000000u);
}

__device__ __forceinline__ float q4_code_plus128_rt(uint32_t word, int k) {
  uint32_t v = (k <= 4) ? (word << (16 - 4 * k)) : (word >> (4 * k - 16));
  return __uint_as_float((v & 0x000f0000u) | 0x43000000u);
}

__device__ __forceinline__ float sb_scale(uint32_t sb) { return __uint_as_float(sb << 16); }
__device__ __forceinline__ float sb_bias(uint32_t sb) { return __uint_as_float(sb & 0xffff0000u); }

}  // namespace dec

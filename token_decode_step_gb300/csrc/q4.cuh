// Affine 4-bit group-64 decoding shared by the GEMV kernels and the dequant test hook.
//
// Format (oxinfer crate page, "MLX checkpoints"): eight 4-bit codes q per uint32,
// one bf16 scale s and bias b per group of 64 inputs, w = s*q + b.  Code k of a
// word sits in bits 4k..4k+3.  The handle stores (s, b) of a (row, group) as one
// uint32: s in the low 16 bits, b in the high 16 bits.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

// Two codes at bits s..s+3 and s+16..s+19 -> f16x2 (q_lo, q_hi), exact: the codes are
// masked into the low mantissa bits of 1024.0 (f16 0x6400, mantissa unit 1), then 1024
// is subtracted.  Used by the batched tensor-core path (A operand) and its dequant hook.
__device__ __forceinline__ uint32_t q4_pair_f16(uint32_t word, int shift) {
  const uint32_t v = ((word >> shift) & 0x000f000fu) | 0x64006400u;
  const __half2 h = *reinterpret_cast<const __half2*>(&v);
  const __half2 off = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
  const __half2 q = __hsub2(h, off);
  return *reinterpret_cast<const uint32_t*>(&q);
}

// The same for bf16: the codes sit in the low mantissa bits of 128.0 (bf16 0x4300,
// mantissa unit 1), then 128 is subtracted; q in 0..15 is exact in bf16.
__device__ __forceinline__ uint32_t q4_pair_bf16(uint32_t word, int shift) {
  const uint32_t v = ((word >> shift) & 0x000f000fu) | 0x43004300u;
  const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&v);
  const __nv_bfloat162 off = __halves2bfloat162(__ushort_as_bfloat16(0x4300), __ushort_as_bfloat16(0x4300));
  const __nv_bfloat162 q = __hsub2(h, off);
  return *reinterpret_cast<const uint32_t*>(&q);
}

__device__ __forceinline__ float sb_scale(uint32_t sb) { return __uint_as_float(sb << 16); }
__device__ __forceinline__ float sb_bias(uint32_t sb) { return __uint_as_float(sb & 0xffff0000u); }

}  // namespace dec

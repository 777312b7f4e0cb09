// Helpers of the batch-1 GEMV kernel (k_gemv1.cu): the input chunk with the
// folded norm weight, the bf16 and affine 4-bit dot products of one chunk, SiLU, and the
// warp sum of eight row sums at once.
#pragma once

#include "dec_internal.cuh"
#include "q4.cuh"

namespace dec {
namespace gemv {

// Input chunk: x[col .. col + n) as floats, times the norm weight for kInNorm.
template <int IN, int N>
__device__ __forceinline__ void load_x(const GemvParams& p, int col, float (&xv)[N]) {
  const float4* src = reinterpret_cast<const float4*>(p.x + col);
#pragma unroll
  for (int i = 0; i < N / 4; ++i) {
    float4 v = src[i];
    xv[4 * i + 0] = v.x;
    xv[4 * i + 1] = v.y;
    xv[4 * i + 2] = v.z;
    xv[4 * i + 3] = v.w;
  }
  if constexpr (IN == kInNorm) {
    const uint4* wn = reinterpret_cast<const uint4*>(p.norm_w + col);
#pragma unroll
    for (int i = 0; i < N / 8; ++i) {
      uint4 u = wn[i];
      xv[8 * i + 0] *= bf16_lo(u.x);
      xv[8 * i + 1] *= bf16_hi(u.x);
      xv[8 * i + 2] *= bf16_lo(u.y);
      xv[8 * i + 3] *= bf16_hi(u.y);
      xv[8 * i + 4] *= bf16_lo(u.z);
      xv[8 * i + 5] *= bf16_hi(u.z);
      xv[8 * i + 6] *= bf16_lo(u.w);
      xv[8 * i + 7] *= bf16_hi(u.w);
    }
  }
}

__device__ __forceinline__ float dot_bf16x8(uint4 w, const float* x, float acc) {
  acc = fmaf(bf16_lo(w.x), x[0], acc);
  acc = fmaf(bf16_hi(w.x), x[1], acc);
  acc = fmaf(bf16_lo(w.y), x[2], acc);
  acc = fmaf(bf16_hi(w.y), x[3], acc);
  acc = fmaf(bf16_lo(w.z), x[4], acc);
  acc = fmaf(bf16_hi(w.z), x[5], acc);
  acc = fmaf(bf16_lo(w.w), x[6], acc);
  acc = fmaf(bf16_hi(w.w), x[7], acc);
  return acc;
}

// (d0, d1) += (a0 * x0, a1 * x1) with one packed fp32 FMA; a0, a1 are float bit patterns
__device__ __forceinline__ void ffma2(float& d0, float& d1, uint32_t a0, uint32_t a1, float x0, float x1) {
  asm("{\n\t.reg .b64 a, x, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 x, {%4, %5};\n\t"
      "mov.b64 d, {%0, %1};\n\t"
      "fma.rn.f32x2 d, a, x, d;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "r"(a0), "r"(a1), "f"(x0), "f"(x1));
}

// (d0, d1) += sum over the 8 codes of one word of (128 + q_k) x_k: even codes in d0,
// odd codes in d1.  Byte j of `lo` is code 2j, byte j of `hi` code 2j + 1; the permute
// selector 0x7j44 builds [0, 0, byte j, 0x43] = 128 + code as a float.
__device__ __forceinline__ void dot_q4_word(uint32_t w, const float* x, float& d0, float& d1) {
  const uint32_t lo = w & 0x0f0f0f0fu, hi = (w >> 4) & 0x0f0f0f0fu;
  constexpr uint32_t kMagic = 0x43000000u;
  ffma2(d0, d1, __byte_perm(lo, kMagic, 0x7044), __byte_perm(hi, kMagic, 0x7044), x[0], x[1]);
  ffma2(d0, d1, __byte_perm(lo, kMagic, 0x7144), __byte_perm(hi, kMagic, 0x7144), x[2], x[3]);
  ffma2(d0, d1, __byte_perm(lo, kMagic, 0x7244), __byte_perm(hi, kMagic, 0x7244), x[4], x[5]);
  ffma2(d0, d1, __byte_perm(lo, kMagic, 0x7344), __byte_perm(hi, kMagic, 0x7344), x[6], x[7]);
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// Warp sums of 8 values at once by halving exchanges: after the xor-16, -8 and -4 steps
// each lane holds a partial of value (lane >> 2) & 7 only, then xor-2 and xor-1 finish
// it (9 shuffles instead of 40).  Every lane returns the full sum of its value; the sum
// order is fixed.
__device__ __forceinline__ float warp_sum8(const float (&v)[8], int lane) {
  float a[4], b[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? v[i + 4] : v[i], send = b4 ? v[i] : v[i + 4];
    a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? a[i + 2] : a[i], send = b3 ? a[i] : a[i + 2];
    b[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float c = (b2 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, b2 ? b[0] : b[1], 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

}  // namespace gemv
}  // namespace dec

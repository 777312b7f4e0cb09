// The unit epilogue of the batched tcgen05 decode projections (k_gemm_q4tc.cu, k_gemm_btc.cu):
// the thread holds weight row n of a tile (128 rows, or 120 in the 4-bit kernel) and its results
// for TPT of the token columns.  When S > 1 pieces of the tile's K range were computed apart (K
// splits, or the segments of a stream-K schedule), the partial results go to p.partials slot
// `split` and the last CTA to finish the tile adds them in slot order; then the input RMSNorm's
// per-token 1/rms and the fused epilogue (store / residual + next-norm hi/lo planes + sums of
// squares / SwiGLU / lm_head keys).  Called by the kernel's NTH epilogue threads together (named
// barrier 1).
#pragma once

#include "dec_internal.cuh"

namespace dec {
namespace tcdec {

// Stream-K schedule of the bf16 kernel: the n_tiles x (K / 64) stages, tile-major, are dealt
// to `grid` CTAs in contiguous ranges [sk_begin(c), sk_begin(c + 1)); sk_cta_of(s) is the CTA
// whose range holds stage s.  A tile's stages then fall to consecutive CTAs, one segment each.
__host__ __device__ inline long long sk_begin(long long c, long long total, long long grid) {
  return c * total / grid;
}
__host__ __device__ inline int sk_cta_of(long long s, long long total, long long grid) {
  return static_cast<int>(((s + 1) * grid + total - 1) / total) - 1;
}

constexpr int kT = 32;  // token columns

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }
template <int NTH = 128>
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NTH) : "memory");
}
__device__ __forceinline__ void split_hl(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// The split exchange in two halves, for a kernel that defers the second past the start of its
// next unit: split_write stores this unit's partial results (slot `split`); split_finish, later,
// takes the tile's ticket and, in the last CTA to arrive, leaves the slots' sum (in slot order)
// in y and returns true.  Called by the NTH epilogue threads together.
template <int TPT>
__device__ __forceinline__ void split_write(const Q4tcParams& p, const float (&y)[TPT], int t0, int n, int split,
                                            bool live) {
  if (live) {
#pragma unroll
    for (int i = 0; i < TPT; ++i)
      if (t0 + i < p.M) p.partials[(static_cast<size_t>(split) * p.M + t0 + i) * p.N + n] = y[i];
  }
}
template <int TPT, int NTH>
__device__ __forceinline__ bool split_finish(const Q4tcParams& p, float (&y)[TPT], int t0, int n, int tile, int S,
                                             bool live, int et, unsigned* s_ticket) {
  __threadfence();
  epi_sync<NTH>();
  if (et == 0) *s_ticket = atomicAdd(&p.counters[tile], 1u);
  epi_sync<NTH>();
  if (*s_ticket != static_cast<unsigned>(S - 1)) return false;
  __threadfence();
#pragma unroll
  for (int i = 0; i < TPT; ++i) y[i] = 0.f;
  if (live)
    for (int s = 0; s < S; ++s)
#pragma unroll
      for (int i = 0; i < TPT; ++i)
        if (t0 + i < p.M) y[i] += __ldcg(p.partials + (static_cast<size_t>(s) * p.M + t0 + i) * p.N + n);
  if (et == 0) p.counters[tile] = 0u;
  return true;
}

// The fused epilogue of a tile's complete results y (TPT tokens per thread from token t0).
template <int IN, int EPI, int TPT>
__device__ __forceinline__ void fused_epilogue(const Q4tcParams& p, float (&y)[TPT], int t0, int n, bool live,
                                               int lane, const float* s_inv, unsigned long long* s_best) {
  if constexpr (IN == kInNorm) {
#pragma unroll
    for (int i = 0; i < TPT; ++i) y[i] *= s_inv[t0 + i];
  }
  if constexpr (EPI == kEpiStore) {
    if (live) {
#pragma unroll
      for (int i = 0; i < TPT; ++i)
        if (t0 + i < p.M) p.out[static_cast<size_t>(t0 + i) * p.N + n] = y[i];
    }
  } else if constexpr (EPI == kEpiResid) {
    // h += y; the next consumer's input h * next_norm as hi, lo planes; sums of squares per
    // 8 rows (lanes 8 j .. 8 j + 7; N is a multiple of 8, so all of them are live or none)
    const float nw = live ? bf16_to_f(p.next_norm_w[n]) : 0.f;
    const size_t plane = static_cast<size_t>(p.M) * p.N;
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      const int t = t0 + i;
      float hn = 0.f;
      const bool on = live && t < p.M;
      if (on) {
        const size_t o = static_cast<size_t>(t) * p.N + n;
        hn = p.out[o] + y[i];
        p.out[o] = hn;
        __nv_bfloat16 hi, lo;
        split_hl(hn * nw, hi, lo);
        p.xhl_out[o] = hi;
        p.xhl_out[plane + o] = lo;
      }
      float ss = hn * hn;
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      ss += __shfl_xor_sync(0xffffffffu, ss, 4);
      if (on && (lane & 7) == 0) p.sumsq_out[static_cast<size_t>(t) * (p.N / kResGroup) + n / kResGroup] = ss;
    }
  } else if constexpr (EPI == kEpiSwiglu) {
    // packed rows in blocks of 4: rows 8 j .. 8 j + 3 gate outputs 4 j .. 4 j + 3, the
    // next 4 rows the matching up outputs (lane ^ 4)
    const size_t plane = static_cast<size_t>(p.M) * (p.N / 2);
    const int o = (n >> 3) * 4 + (n & 3);
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      const int t = t0 + i;
      const float up = __shfl_xor_sync(0xffffffffu, y[i], 4);
      if (live && (n & 4) == 0 && t < p.M) {
        const float gv = silu(y[i]) * up;
        const size_t oo = static_cast<size_t>(t) * (p.N / 2) + o;
        p.out[oo] = gv;
        __nv_bfloat16 hi, lo;
        split_hl(gv, hi, lo);
        p.xhl_out[oo] = hi;
        p.xhl_out[plane + oo] = lo;
      }
    }
  } else {  // lm_head: logits, and every token's best (value, index) key over the warp's rows
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      const int t = t0 + i;
      const bool on = live && t < p.M;
      if (on && p.out) p.out[static_cast<size_t>(t) * p.N + n] = y[i];
      unsigned long long k = on ? argmax_key(y[i], n) : 0ull;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, k, o);
        k = other > k ? other : k;
      }
      if (lane == 0 && k != 0ull) atomicMax(s_best + t, k);
    }
  }
}

// Both: TPT tokens per thread, starting at token t0 (the thread's accumulator columns); NTH
// epilogue threads take part in the named barrier.
template <int IN, int EPI, int TPT, int NTH>
__device__ __forceinline__ void unit_epilogue(const Q4tcParams& p, float (&y)[TPT], int t0, int n, int tile,
                                              int split, int S, bool live, int et, int lane, const float* s_inv,
                                              unsigned long long* s_best, unsigned* s_ticket) {
  if (S > 1) {  // partial results; the last CTA of the tile adds them in slot order
    split_write<TPT>(p, y, t0, n, split, live);
    if (!split_finish<TPT, NTH>(p, y, t0, n, tile, S, live, et, s_ticket)) return;
  }
  fused_epilogue<IN, EPI, TPT>(p, y, t0, n, live, lane, s_inv, s_best);
}

}  // namespace tcdec
}  // namespace dec

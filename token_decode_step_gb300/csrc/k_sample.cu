// On-device sampling of the next token from the lm_head logits, one CTA per row:
// temperature, top-k, top-p, then an inverse-CDF draw; temperature 0 is the argmax.
//
// Source: Butter architecture.md, section on GPU sampling (the final kernel of the
// per-token command buffer: logits times 1/temp, top-k by sorting the k largest,
// top-p by a cumulative-softmax threshold, an inverse-CDF sample with an RNG state,
// a 4-byte token id as the only output).
//
// Steps in a CTA of 1024 threads:
//  1. order keys: every float32 logit maps to a uint32 whose unsigned order is the
//     float order (-0 taken as +0, NaN below everything);
//  2. the k-th largest key by a 4-pass radix select (8-bit digits, shared-memory
//     histograms over the row);
//  3. the k candidates: keys above the threshold, then threshold ties in index order;
//  4. a bitonic sort of (key, index) into (logit descending, index ascending);
//  5. p_j = exp((l_j - l_0) / T), an inclusive scan in a fixed order, the top-p prefix,
//     and the first kept candidate whose cumulative mass exceeds u times the prefix
//     mass, u from Philox4x32-10 (the published counter-based generator: ten rounds of
//     two 32x32->64 multiplies with Weyl-sequence round keys).
#include "dec_internal.cuh"

namespace dec {

namespace {

constexpr int kSampleThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN
  if ((b & 0x7fffffffu) == 0u) b = 0u;             // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Philox4x32-10: returns the first output word for (counter, key).
__device__ uint32_t philox_first(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u, kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(kM0, c0), lo0 = kM0 * c0;
    const uint32_t hi1 = __umulhi(kM1, c2), lo1 = kM1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += kW0;
    k1 += kW1;
  }
  return c0;
}

// inclusive scan over the CTA (one value per thread, fixed association order)
__device__ float block_scan(float v, float* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    warp_tot[lane] = t;  // inclusive totals of warps 0..lane
  }
  __syncthreads();
  return warp > 0 ? v + warp_tot[warp - 1] : v;
}

__global__ void __launch_bounds__(kSampleThreads) k_sample(SampleParams p) {
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* lg = p.logits + static_cast<size_t>(row) * p.V;
  __shared__ unsigned hist[256];
  __shared__ unsigned long long cand[kSampleThreads];  // (key << 32) | (~index)
  __shared__ float warp_tot[32];
  __shared__ unsigned warp_cnt[32];
  __shared__ unsigned s_prefix, s_remaining, s_ngt, s_eq_base;
  __shared__ int s_m, s_token;
  __shared__ unsigned long long s_best[32];

  if (!(p.temperature > 0.f)) {  // greedy: the argmax, lowest index on ties
    unsigned long long best = 0ull;
    for (int i = tid; i < p.V; i += kSampleThreads) {
      const unsigned long long c = (static_cast<unsigned long long>(order_key(lg[i])) << 32) | (0xffffffffu - i);
      best = c > best ? c : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long n = __shfl_xor_sync(0xffffffffu, best, o);
      best = n > best ? n : best;
    }
    if (lane == 0) s_best[warp] = best;
    __syncthreads();
    if (tid == 0) {
      unsigned long long b = 0ull;
      for (int w = 0; w < kSampleThreads / 32; ++w) b = s_best[w] > b ? s_best[w] : b;
      p.tokens[row] = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(b));
    }
    return;
  }

  int k = (p.top_k >= 1 && p.top_k <= kSampleMaxK) ? p.top_k : kSampleMaxK;
  k = k < p.V ? k : p.V;

  // ---- 2. radix select of the k-th largest key
  if (tid == 0) {
    s_prefix = 0u;
    s_remaining = static_cast<unsigned>(k);
  }
  unsigned mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSampleThreads) hist[i] = 0u;
    __syncthreads();
    const unsigned prefix = s_prefix;
    for (int i = tid; i < p.V; i += kSampleThreads) {
      const uint32_t key = order_key(lg[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {  // the digit where the count from the top reaches the remaining rank
      unsigned above = 0u, rem = s_remaining;
      int d = 255;
      for (; d > 0; --d) {
        if (above + hist[d] >= rem) break;
        above += hist[d];
      }
      s_prefix = prefix | (static_cast<unsigned>(d) << shift);
      s_remaining = rem - above;
    }
    mask |= 0xffu << shift;
    __syncthreads();
  }
  const uint32_t thr = s_prefix;
  const unsigned need_eq = s_remaining;  // ties at the threshold taken, lowest indices first

  // ---- 3. gather: keys above the threshold (any order), ties in index order
  if (tid == 0) {
    s_ngt = 0u;
    s_eq_base = 0u;
  }
  cand[tid] = 0ull;
  __syncthreads();
  const unsigned ngt_total = static_cast<unsigned>(k) - need_eq;
  for (int base = 0; base < p.V; base += kSampleThreads) {
    const int i = base + tid;
    const uint32_t key = i < p.V ? order_key(lg[i]) : 0u;
    const bool gt = i < p.V && key > thr, eq = i < p.V && key == thr;
    const unsigned long long c = (static_cast<unsigned long long>(key) << 32) | (0xffffffffu - i);
    if (gt) cand[atomicAdd(&s_ngt, 1u)] = c;
    const unsigned bal = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) warp_cnt[warp] = __popc(bal);
    __syncthreads();
    unsigned before = s_eq_base;
    for (int w = 0; w < warp; ++w) before += warp_cnt[w];
    before += __popc(bal & ((1u << lane) - 1u));
    if (eq && before < need_eq) cand[ngt_total + before] = c;
    __syncthreads();
    if (tid == 0) {
      unsigned t = 0u;
      for (int w = 0; w < kSampleThreads / 32; ++w) t += warp_cnt[w];
      s_eq_base += t;
    }
    __syncthreads();
    if (s_eq_base >= need_eq && s_ngt >= ngt_total) break;  // uniform: shared values after a barrier
  }

  // ---- 4. bitonic sort, descending (logit descending, then index ascending)
  int P = 1;
  while (P < k) P <<= 1;
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      const int i = tid, j = tid ^ stride;
      if (i < P && j > i) {
        const unsigned long long a = cand[i], b = cand[j];
        const bool desc = (i & size) == 0;
        if (desc ? (a < b) : (a > b)) {
          cand[i] = b;
          cand[j] = a;
        }
      }
    }
  }
  __syncthreads();

  // ---- 5. probabilities, prefix sums, top-p cut, draw
  const float l0 = key_value(static_cast<uint32_t>(cand[0] >> 32));
  float pj = 0.f;
  if (tid < k) pj = expf((key_value(static_cast<uint32_t>(cand[tid] >> 32)) - l0) / p.temperature);
  const float cum = block_scan(pj, warp_tot);
  __shared__ float s_cum[kSampleThreads];
  s_cum[tid] = cum;
  if (tid == 0) s_m = k;
  __syncthreads();
  if (p.top_p < 1.f) {
    const float cut = p.top_p * s_cum[k - 1];
    if (tid < k && cum >= cut && (tid == 0 || s_cum[tid - 1] < cut)) s_m = tid + 1;
    __syncthreads();
  }
  const int m = s_m;
  if (tid == 0) {
    const unsigned long long off = p.offset_dev ? *p.offset_dev : p.offset;
    const uint32_t x0 = philox_first(static_cast<uint32_t>(off), static_cast<uint32_t>(off >> 32),
                                     static_cast<uint32_t>(row), 0u, static_cast<uint32_t>(p.seed),
                                     static_cast<uint32_t>(p.seed >> 32));
    warp_tot[0] = static_cast<float>(x0 >> 8) * 0x1p-24f * s_cum[m - 1];  // the draw target
    s_token = static_cast<int>(0xffffffffu - static_cast<uint32_t>(cand[m - 1]));  // if rounding leaves none
  }
  __syncthreads();
  const float target = warp_tot[0];
  if (tid < m && cum > target && (tid == 0 || s_cum[tid - 1] <= target))
    s_token = static_cast<int>(0xffffffffu - static_cast<uint32_t>(cand[tid]));
  __syncthreads();
  if (tid == 0) p.tokens[row] = s_token;
}

}  // namespace

cudaError_t launch_sample(cudaStream_t s, const SampleParams& p, int batch) {
  k_sample<<<batch, kSampleThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dec

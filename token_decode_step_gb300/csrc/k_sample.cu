// On-device sampling of the next token from the lm_head logits, one CTA per row:
// temperature, top-k, top-p, then an inverse-CDF draw; temperature 0 is the argmax.
//
// Source: Butter architecture.md, section on GPU sampling (the final kernel of the
// per-token command buffer: logits times 1/temp, top-k by sorting the k largest,
// top-p by a cumulative-softmax threshold, an inverse-CDF sample with an RNG state,
// a 4-byte token id as the only output).
//
// Steps, for one row per 8-CTA thread-block cluster of 1024 threads each (CTA r scans
// 1/8 of the row; counts and candidates meet in rank 0's shared memory):
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
constexpr int kSampleCluster = 8;  // CTAs per row

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN
  if ((b & 0x7fffffffu) == 0u) b = 0u;             // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

constexpr int kSampleUnroll = 8;   // loads in flight per thread in each pass over a row

// keys of elements base + u * kSampleThreads + threadIdx.x, u < kSampleUnroll (0 past the end):
// all loads issued before any is used
__device__ __forceinline__ void load_keys(const float* lg, int V, int base, uint32_t (&keys)[kSampleUnroll]) {
  float v[kSampleUnroll];
#pragma unroll
  for (int u = 0; u < kSampleUnroll; ++u) {
    const int i = base + u * kSampleThreads + static_cast<int>(threadIdx.x);
    v[u] = i < V ? __ldg(lg + i) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < kSampleUnroll; ++u) {
    const int i = base + u * kSampleThreads + static_cast<int>(threadIdx.x);
    keys[u] = i < V ? order_key(v[u]) : 0u;
  }
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

// shared::cluster helpers (rank 0 holds the row's histograms and candidates)
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_map(const void* smem_ptr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(smem_ptr)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_red_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t cl_atom_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void cl_st_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void cl_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t cl_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// One row per thread-block cluster of kSampleCluster CTAs: CTA r scans the contiguous
// slice [r per, (r + 1) per) of the row; the histograms, the selection state and the
// candidates live in rank 0's shared memory, which finishes the row alone.
__global__ void __launch_bounds__(kSampleThreads) k_sample(SampleParams p) {
  const int row = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cl_rank();
  const float* lg = p.logits + static_cast<size_t>(row) * p.V;
  const int per = (p.V + kSampleCluster - 1) / kSampleCluster;
  const int lo = static_cast<int>(rank) * per, hi = min(p.V, lo + per);

  __shared__ unsigned hist[256];
  __shared__ unsigned ghist[4][256];                   // rank 0: the cluster's histogram per pass
  __shared__ unsigned long long cand[kSampleThreads];  // rank 0: (key << 32) | (~index)
  __shared__ unsigned long long best_all[kSampleCluster];  // rank 0: greedy, per CTA
  __shared__ unsigned eq_cnt[kSampleCluster];          // rank 0: threshold ties per CTA
  __shared__ float warp_tot[32];
  __shared__ unsigned warp_cnt[32];
  __shared__ unsigned s_prefix, s_remaining, s_count_eq, s_slot, s_eq_base;  // rank 0's are the cluster's
  __shared__ int s_m, s_token;
  __shared__ unsigned long long s_best[32];
  __shared__ float s_cum[kSampleThreads];

  // rank 0 clears its cluster state, then the first barrier (also: every CTA is running
  // before any remote access)
  if (rank == 0) {
    for (int i = tid; i < 4 * 256; i += kSampleThreads) (&ghist[0][0])[i] = 0u;
    if (tid == 0) s_slot = 0u;
  }
  cand[tid] = 0ull;
  cl_sync();
  const uint32_t r0 = 0u;

  if (!(p.temperature > 0.f)) {  // greedy: the argmax, lowest index on ties
    unsigned long long best = 0ull;
    for (int base = lo; base < hi; base += kSampleThreads * kSampleUnroll) {
      uint32_t keys[kSampleUnroll];
      load_keys(lg, hi, base, keys);
#pragma unroll
      for (int u = 0; u < kSampleUnroll; ++u) {
        const int i = base + u * kSampleThreads + tid;
        const unsigned long long c = (static_cast<unsigned long long>(keys[u]) << 32) | (0xffffffffu - i);
        if (i < hi) best = c > best ? c : best;
      }
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
      cl_st_u64(cl_map(&best_all[rank], r0), b);
    }
    cl_sync();
    if (rank == 0 && tid == 0) {
      unsigned long long b = 0ull;
      for (int r = 0; r < kSampleCluster; ++r) b = best_all[r] > b ? best_all[r] : b;
      p.tokens[row] = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(b));
    }
    return;
  }

  int k = (p.top_k >= 1 && p.top_k <= kSampleMaxK) ? p.top_k : kSampleMaxK;
  k = k < p.V ? k : p.V;

  // ---- 2. radix select of the k-th largest key over the cluster
  unsigned prefix = 0u, remaining = static_cast<unsigned>(k), count_eq = 0u, mask = 0u;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kSampleThreads) hist[i] = 0u;
    __syncthreads();
    for (int base = lo; base < hi; base += kSampleThreads * kSampleUnroll) {
      uint32_t keys[kSampleUnroll];
      load_keys(lg, hi, base, keys);
#pragma unroll
      for (int u = 0; u < kSampleUnroll; ++u) {
        // lanes with the same digit add once (logits crowd a few bins: unaggregated
        // shared atomics on one address serialise)
        const int i = base + u * kSampleThreads + tid;
        const bool in = i < hi && (keys[u] & mask) == prefix;
        const unsigned digit = in ? (keys[u] >> shift) & 255u : 256u;
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], static_cast<unsigned>(__popc(peers)));
      }
    }
    __syncthreads();
    if (tid < 256 && hist[tid]) cl_red_add(cl_map(&ghist[pass][tid], r0), hist[tid]);
    cl_sync();
    if (rank == 0 && tid == 0) {  // the digit where the count from the top reaches the remaining rank
      unsigned above = 0u;
      int d = 255;
      for (; d > 0; --d) {
        if (above + ghist[pass][d] >= remaining) break;
        above += ghist[pass][d];
      }
      s_prefix = prefix | (static_cast<unsigned>(d) << shift);
      s_remaining = remaining - above;
      s_count_eq = ghist[pass][d];  // after the last pass: the elements equal to the threshold
    }
    cl_sync();
    prefix = cl_ld_u32(cl_map(&s_prefix, r0));
    remaining = cl_ld_u32(cl_map(&s_remaining, r0));
    count_eq = cl_ld_u32(cl_map(&s_count_eq, r0));
    mask |= 0xffu << shift;
  }
  const uint32_t thr = prefix;
  const unsigned need_eq = remaining;  // ties at the threshold taken, lowest indices first
  const unsigned ngt_total = static_cast<unsigned>(k) - need_eq;
  const uint32_t slot_addr = cl_map(&s_slot, r0);

  // ---- 3. gather into rank 0: keys above the threshold (any slot), ties in index order
  if (count_eq == need_eq) {  // every tie is kept: slots by an atomic counter (the sort fixes the order)
    for (int base = lo; base < hi; base += kSampleThreads * kSampleUnroll) {
      uint32_t keys[kSampleUnroll];
      load_keys(lg, hi, base, keys);
#pragma unroll
      for (int u = 0; u < kSampleUnroll; ++u) {
        const int i = base + u * kSampleThreads + tid;
        if (i < hi && keys[u] >= thr) {
          const uint32_t slot = cl_atom_add(slot_addr, 1u);
          cl_st_u64(cl_map(&cand[slot], r0), (static_cast<unsigned long long>(keys[u]) << 32) | (0xffffffffu - i));
        }
      }
    }
  } else {  // ties straddle the k-th place: the lowest indices among them, slices in rank order
    unsigned my_eq = 0u;
    for (int i = lo + tid; i < hi; i += kSampleThreads) my_eq += order_key(lg[i]) == thr ? 1u : 0u;
    my_eq = __reduce_add_sync(0xffffffffu, my_eq);
    if (lane == 0) warp_cnt[warp] = my_eq;
    __syncthreads();
    if (tid == 0) {
      unsigned t = 0u;
      for (int w = 0; w < kSampleThreads / 32; ++w) t += warp_cnt[w];
      cl_st_u32(cl_map(&eq_cnt[rank], r0), t);
    }
    cl_sync();
    if (tid == 0) {
      unsigned b = 0u;
      for (uint32_t r = 0; r < rank; ++r) b += cl_ld_u32(cl_map(&eq_cnt[r], r0));
      s_eq_base = b;
    }
    __syncthreads();
    for (int base = lo; base < hi; base += kSampleThreads) {
      const int i = base + tid;
      const uint32_t key = i < hi ? order_key(lg[i]) : 0u;
      const bool gt = i < hi && key > thr, eq = i < hi && key == thr;
      const unsigned long long c = (static_cast<unsigned long long>(key) << 32) | (0xffffffffu - i);
      if (gt) cl_st_u64(cl_map(&cand[cl_atom_add(slot_addr, 1u)], r0), c);
      const unsigned bal = __ballot_sync(0xffffffffu, eq);
      if (lane == 0) warp_cnt[warp] = __popc(bal);
      __syncthreads();
      unsigned before = s_eq_base;
      for (int w = 0; w < warp; ++w) before += warp_cnt[w];
      before += __popc(bal & ((1u << lane) - 1u));
      if (eq && before < need_eq) cl_st_u64(cl_map(&cand[ngt_total + before], r0), c);
      __syncthreads();
      if (tid == 0) {
        unsigned t = 0u;
        for (int w = 0; w < kSampleThreads / 32; ++w) t += warp_cnt[w];
        s_eq_base += t;
      }
      __syncthreads();
    }
  }
  cl_sync();  // every candidate is in rank 0; no remote access follows
  if (rank != 0) return;

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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSampleCluster, batch);
  cfg.blockDim = dim3(kSampleThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSampleCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_sample, p);
}

}  // namespace dec

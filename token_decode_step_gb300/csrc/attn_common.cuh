// Pieces shared by the decode-attention kernels of both KV cache formats (bf16 rows and
// affine 8-bit codes): thread-block-cluster helpers, the split of a sequence's positions
// over the cluster's CTAs, the cluster merge of the partial softmax results, and the
// launch-shape plumbing (cluster sizes, ring depths, occupancy of each shape).
#pragma once

#include "dec_internal.cuh"

namespace dec {
namespace attn {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// split form: arrive early without ordering memory, wait before the first remote access
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared-memory address of the same variable in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t map_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Positions [begin, end) of CTA `rank` of a cluster of C for a sequence with T = P + 1
// positions: runs of ceil(T / C) rounded up to 16 positions; later CTAs may get fewer
// or none.
__device__ __forceinline__ void attention_run(int T, int C, int rank, int* begin, int* end) {
  const int per = (T + C - 1) / C;
  const int len = (per + 15) / 16 * 16;
  const int b0 = rank * len;
  *begin = b0 < T ? b0 : T;
  *end = b0 + len < T ? b0 + len : T;
}

// Receive area of the cluster merge: up to 16 records of (m[G], l[G], acc[ceil(G D / C)]), G <= 4.
template <int D>
struct Xchg {
  static constexpr int kFloats = 16 * 2 * 4 + 4 * D + 16;
};

// The merge, after each warp left its state in shared memory: mw[4][G] running maxima
// (exp2 domain), lw[4][G] sums, ow[4][G][D] un-normalised outputs.  Pushed through
// distributed shared memory: CTA `rank` owns outputs [rank kPer, (rank + 1) kPer) of the
// G D; every CTA combines its four warps, stores its (m, l) per head and its combined
// partial outputs of each owner's slice into the owner's receive area (record `rank`:
// m[G], l[G], acc[kPer]), then one cluster barrier, then each owner merges from its own
// memory and writes out[b][h G D + i] (and the hi / lo planes of the batched path).  The
// first cluster barrier phase (arrived at kernel start) is waited for before the first
// remote store, so every CTA of the cluster is known to be running.
template <int D, int G, int C>
__device__ __forceinline__ void merge_store(const AttnParams& p, const float* mw, const float* lw, const float* ow,
                                            float* xchg, float* fw, int rank, int b, int h, int tid) {
  constexpr int kOut = G * D;
  constexpr int kPer = (kOut + C - 1) / C;
  constexpr int kRec = 2 * G + kPer;
  static_assert(C * kRec <= Xchg<D>::kFloats, "receive area too small");
  const uint32_t recv_local = smem_u32(xchg);
  cluster_wait();
  if (tid < G) {
    float M = -INFINITY;
    for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * G + tid]);
    float L = 0.f;
    for (int w = 0; w < 4; ++w) {
      const float f = (M == -INFINITY) ? 0.f : exp2f(mw[w * G + tid] - M);
      fw[w * G + tid] = f;
      L += f * lw[w * G + tid];
    }
#pragma unroll 1
    for (int r = 0; r < C; ++r) {
      const uint32_t rec = map_rank(recv_local + (rank * kRec) * 4, static_cast<uint32_t>(r));
      st_cluster_f32(rec + tid * 4, M);
      st_cluster_f32(rec + (G + tid) * 4, L);
    }
  }
  __syncthreads();
  for (int i = tid; i < kOut; i += kAttnThreads) {
    const int j = i / D, e = i % D;
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) a += fw[w * G + j] * ow[(w * G + j) * D + e];
    const int owner = i / kPer;
    const uint32_t rec = map_rank(recv_local + (rank * kRec) * 4, static_cast<uint32_t>(owner));
    st_cluster_f32(rec + (2 * G + i - owner * kPer) * 4, a);
  }
  cluster_sync();
  float* out_b = p.out + static_cast<size_t>(b) * p.nq * D + h * G * D;
  const int i_end = (rank + 1) * kPer < kOut ? (rank + 1) * kPer : kOut;
  for (int i = rank * kPer + tid; i < i_end; i += kAttnThreads) {
    const int j = i / D, k = i - rank * kPer;
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < C; ++r) M = fmaxf(M, xchg[r * kRec + j]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int r = 0; r < C; ++r) {
      const float mr = xchg[r * kRec + j];
      const float f = (mr == -INFINITY) ? 0.f : exp2f(mr - M);
      num = fmaf(f, xchg[r * kRec + 2 * G + k], num);
      den = fmaf(f, xchg[r * kRec + G + j], den);
    }
    const float ov = num / den;
    out_b[i] = ov;
    if (p.out_hl) {  // batched path: the O projection's input as hi + lo planes
      const size_t o = static_cast<size_t>(b) * p.nq * D + h * G * D + i;
      const __nv_bfloat16 hi = __float2bfloat16_rn(ov);
      p.out_hl[o] = hi;
      p.out_hl[static_cast<size_t>(p.B) * p.nq * D + o] = __float2bfloat16_rn(ov - __bfloat162float(hi));
    }
  }
  // no shared::cluster access follows the barrier: CTAs leave independently
}

// ---------------------------------------------------------------- launch shapes
// 0 = clusters of 8, shallow ring; 1 = clusters of 8, deep ring; 2 = clusters of 16,
// deep ring; 3 = clusters of 12, deep ring (16 and 12 are non-portable sizes);
// 4 = clusters of 4, shallow ring.  KT<D, G, C, DEEP> names a kernel (KT::kernel()) and
// its dynamic shared memory (KT::kSmem).
constexpr int kShapes = 5;

template <template <int, int, int, bool> class KT, int D, int G, int C, bool DEEP>
cudaLaunchConfig_t config(const AttnParams& p, cudaStream_t stream, bool pdl, cudaLaunchAttribute (&attr)[2]) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, p.nkv, p.B);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = KT<D, G, C, DEEP>::kSmem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <template <int, int, int, bool> class KT, int D, int G, int C, bool DEEP>
cudaError_t launch_t(const LaunchCtx& c, const AttnParams& p) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = config<KT, D, G, C, DEEP>(p, c.stream, c.pdl, attr);
  return cudaLaunchKernelEx(&cfg, KT<D, G, C, DEEP>::kernel(), p);
}

// Shared-memory limit (and the non-portable cluster size), then the number of
// clusters of this shape that fit on the device at once.
template <template <int, int, int, bool> class KT, int D, int G, int C, bool DEEP>
cudaError_t prepare_t(int* max_clusters) {
  auto kern = KT<D, G, C, DEEP>::kernel();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(KT<D, G, C, DEEP>::kSmem));
  if (e != cudaSuccess) return e;
  if (C > 8 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return e;
  AttnParams probe = {};
  probe.B = 1;
  probe.nkv = 1;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = config<KT, D, G, C, DEEP>(probe, nullptr, false, attr);
  cfg.numAttrs = 1;  // the cluster dimension only
  return cudaOccupancyMaxActiveClusters(max_clusters, kern, &cfg);
}

template <template <int, int, int, bool> class KT, int D, int G>
cudaError_t prepare_all(int (&max_clusters)[kShapes]) {
  cudaError_t e;
  if ((e = prepare_t<KT, D, G, 8, false>(&max_clusters[0])) != cudaSuccess) return e;
  if ((e = prepare_t<KT, D, G, 8, true>(&max_clusters[1])) != cudaSuccess) return e;
  if ((e = prepare_t<KT, D, G, 16, true>(&max_clusters[2])) != cudaSuccess) return e;
  if ((e = prepare_t<KT, D, G, 12, true>(&max_clusters[3])) != cudaSuccess) return e;
  return prepare_t<KT, D, G, 4, false>(&max_clusters[4]);
}

template <template <int, int, int, bool> class KT, int D, int G>
cudaError_t launch_shape(const LaunchCtx& c, const AttnParams& p, int shape) {
  if (shape == 4) return launch_t<KT, D, G, 4, false>(c, p);
  if (shape == 3) return launch_t<KT, D, G, 12, true>(c, p);
  if (shape == 2) return launch_t<KT, D, G, 16, true>(c, p);
  if (shape == 1) return launch_t<KT, D, G, 8, true>(c, p);
  return launch_t<KT, D, G, 8, false>(c, p);
}

// Every (head_dim, group) the kernels are built for: prepare_all / launch_shape of KT.
template <template <int, int, int, bool> class KT>
cudaError_t prepare_dims(int head_dim, int G, int (&max_clusters)[kShapes]) {
#define DEC_ATTN_PREP(D_, G_) \
  if (head_dim == D_ && G == G_) return prepare_all<KT, D_, G_>(max_clusters);
  DEC_ATTN_PREP(64, 1)
  DEC_ATTN_PREP(64, 2)
  DEC_ATTN_PREP(64, 4)
  DEC_ATTN_PREP(128, 1)
  DEC_ATTN_PREP(128, 2)
  DEC_ATTN_PREP(128, 4)
#undef DEC_ATTN_PREP
  return cudaErrorInvalidValue;
}

template <template <int, int, int, bool> class KT>
cudaError_t launch_dims(const LaunchCtx& c, const AttnParams& p, int head_dim, int shape) {
  const int G = p.nq / p.nkv;
#define DEC_ATTN_CASE(D_, G_) \
  if (head_dim == D_ && G == G_) return launch_shape<KT, D_, G_>(c, p, shape);
  DEC_ATTN_CASE(64, 1)
  DEC_ATTN_CASE(64, 2)
  DEC_ATTN_CASE(64, 4)
  DEC_ATTN_CASE(128, 1)
  DEC_ATTN_CASE(128, 2)
  DEC_ATTN_CASE(128, 4)
#undef DEC_ATTN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace attn
}  // namespace dec

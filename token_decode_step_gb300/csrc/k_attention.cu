// Fused decode attention for one layer:
//   per-head RMSNorm of q and k (q_norm / k_norm), rotate-half RoPE at position P,
//   append bf16(k), bf16(v) at cache slot P, then GQA attention of the new token
//   over slots 0..P, split along the positions (flash-decoding) with a
//   log-sum-exp merge of the splits.
//
// Sources: ANEForge "LLMs on the ANE", "Correctness" (QK-norm: per-head RMSNorm
// on Q and K before RoPE) and "What's inside" (RoPE = x cos + rotate_half(x) sin;
// KV heads shared by groups of query heads); Butter architecture.md, "SINGLE-
// TOKEN DECODE" (rope at offset = cache.length, cache.append writes into the
// preallocated buffer, sdpa_decode over the cache).
//
// Grid (C, n_kv, B) in thread-block clusters of C CTAs along x: the cluster of
// (sequence b, KV head h) splits that sequence's T = P+1 positions into C equal
// runs of whole 64-position tiles (so ragged batches stay balanced), CTA r takes
// run r.  Each CTA streams its K/V tiles into shared memory with cp.async
// through a ring of S stages (XOR-swizzled 16-byte chunks so ldmatrix is
// conflict-free; the first S-1 tiles are requested before the grid-dependency
// wait) and runs both products on tensor cores (mma.sync m16n8k16, bf16 in, fp32
// accumulate): the group's G query heads share every K/V row.  q and the
// probabilities enter as bf16 hi + lo rows (rows 0..G-1 and G..2G-1 of the
// 16-row A operand), ~16 significant bits; softmax statistics are fp32 in the
// exp2 domain.  The C partial results are merged through distributed shared
// memory between two cluster barriers: CTA r combines a 1/C slice of the
// outputs from all C CTAs (no global partials, no atomics).
#include "dec_internal.cuh"

namespace dec {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct AttnCfg {
  static constexpr int kStages = D == 128 ? 3 : 4;  // two CTAs per SM (6 stages measured slower when batched)
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = kAttnTile * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;                  // K tile then V tile
  static constexpr int kOffQ = 0;                                      // [16][D] bf16
  static constexpr int kOffStages = 16 * kRowBytes;
  static constexpr int kOffNew = kOffStages + kStages * kStageBytes;  // new k row, new v row
  static constexpr int kOffXchg = kOffNew + 2 * kRowBytes;             // [G][D + 2] floats (G <= 4)
  static constexpr int kOffMisc = kOffXchg + 4 * (D + 2) * 4;          // [4][G] floats
  static constexpr int kBytes = kOffMisc + 64 * 4;
};

// byte offset of 16-byte chunk c of row r inside a swizzled tile
template <int D>
__device__ __forceinline__ int swz(int r, int c) {
  return r * (D * 2) + ((c ^ (r & 7)) << 4);
}

template <int D>
__device__ __forceinline__ void load_tile(uint32_t sdst, const __nv_bfloat16* plane_base, int pos0, int valid_end) {
  constexpr int kChunks = D / 8;
  constexpr int kTotal = kAttnTile * kChunks;
#pragma unroll
  for (int j = 0; j < kTotal / kAttnThreads; ++j) {
    const int idx = threadIdx.x + j * kAttnThreads;
    const int r = idx / kChunks, c = idx % kChunks;
    const int pos = pos0 + r;
    const bool ok = pos < valid_end;
    const __nv_bfloat16* src = plane_base + static_cast<size_t>(ok ? pos : 0) * D + c * 8;
    cp_async16(sdst + swz<D>(r, c), src, ok ? 16 : 0);
  }
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

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

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Positions [begin, end) of CTA `rank` of a cluster of C for a sequence with T = P + 1
// positions: runs of ceil(ceil(T / C) / 64) whole tiles; later CTAs may get none.
__device__ __forceinline__ void attention_run(int T, int C, int rank, int* begin, int* end) {
  const int per = (T + C - 1) / C;
  const int len = (per + kAttnTile - 1) / kAttnTile * kAttnTile;
  const int b0 = rank * len;
  *begin = b0 < T ? b0 : T;
  *end = b0 + len < T ? b0 + len : T;
}

}  // namespace

template <int D, int G, int C>
__global__ void __launch_bounds__(kAttnThreads) k_attention(AttnParams p) {
  using CF = AttnCfg<D>;
  constexpr int S = CF::kStages;
  extern __shared__ __align__(128) unsigned char smem[];

  tl_mark(p.tl, 0);
  const int h = blockIdx.y, b = blockIdx.z;
  const int rank = static_cast<int>(cluster_ctarank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  int P = p.positions[b];
  P = P < 0 ? 0 : (P >= p.max_ctx ? p.max_ctx - 1 : P);  // flagged by the embedding kernel
  const int T = P + 1;
  int pos_begin, pos_end;
  attention_run(T, C, rank, &pos_begin, &pos_end);
  const int ntiles = (pos_end - pos_begin + kAttnTile - 1) / kAttnTile;
  const bool has_new = (P >= pos_begin && P < pos_end);

  const size_t plane = static_cast<size_t>(p.B) * p.nkv * p.max_ctx * D;
  const size_t head_off = (static_cast<size_t>(b) * p.nkv + h) * p.max_ctx * D;
  __nv_bfloat16* kbase = p.kv + (static_cast<size_t>(p.layer) * 2 + 0) * plane + head_off;
  __nv_bfloat16* vbase = p.kv + (static_cast<size_t>(p.layer) * 2 + 1) * plane + head_off;

  const uint32_t s_base = smem_u32(smem);
  const uint32_t sStages = s_base + CF::kOffStages;
  float* xchg = reinterpret_cast<float*>(smem + CF::kOffXchg);  // this CTA's [G][m, l, acc[D]]
  float* misc = reinterpret_cast<float*>(smem + CF::kOffMisc);

  // Cached K/V tiles do not depend on upstream kernels of this step: request the
  // first S-1 before the grid-dependency wait.
#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    if (s < ntiles) {
      const int pos0 = pos_begin + s * kAttnTile;
      load_tile<D>(sStages + s * CF::kStageBytes, kbase, pos0, pos_end);
      load_tile<D>(sStages + s * CF::kStageBytes + CF::kTileBytes, vbase, pos0, pos_end);
    }
    cp_async_commit();
  }
  {  // zero the Q operand (rows 2G..15 stay zero)
    uint32_t* q32 = reinterpret_cast<uint32_t*>(smem + CF::kOffQ);
    for (int i = tid; i < 16 * D / 2; i += kAttnThreads) q32[i] = 0u;
  }

  griddep_wait();
  tl_mark(p.tl, 1);
  __syncthreads();

  float m_run = -INFINITY, l_run = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  if (ntiles > 0) {
    // ---- q/k per-head RMSNorm + RoPE (+ KV append by the CTA holding slot P)
    const int nqkv = (p.nq + 2 * p.nkv) * D;
    const float* qkv_b = p.qkv + static_cast<size_t>(b) * nqkv;
    const float2* rope_b = p.rope + static_cast<size_t>(b) * (D / 2);
    constexpr int E = D / 32;  // elements per lane: lane + 32 m
    auto norm_rope = [&](const float* src, const __nv_bfloat16* wn, float (&y)[E]) {
      float x[E];
      float ss = 0.f;
#pragma unroll
      for (int m = 0; m < E; ++m) {
        x[m] = src[lane + 32 * m];
        ss = fmaf(x[m], x[m], ss);
      }
      ss = warp_sum(ss);
      const float inv = rsqrtf(ss / static_cast<float>(D) + p.eps);
#pragma unroll
      for (int m = 0; m < E; ++m) x[m] = (x[m] * inv) * bf16_to_f(wn[lane + 32 * m]);
      // pairs (e, e + D/2): lane's elements m and m + E/2
#pragma unroll
      for (int m = 0; m < E / 2; ++m) {
        const float2 cs = rope_b[lane + 32 * m];
        const float a = x[m], c = x[m + E / 2];
        y[m] = a * cs.x - c * cs.y;
        y[m + E / 2] = c * cs.x + a * cs.y;
      }
    };
    if (warp < G) {
      float y[E];
      norm_rope(qkv_b + (h * G + warp) * D, p.q_norm, y);
      __nv_bfloat16* q16 = reinterpret_cast<__nv_bfloat16*>(smem + CF::kOffQ);
#pragma unroll
      for (int m = 0; m < E; ++m) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(y[m]);
        const __nv_bfloat16 lo = __float2bfloat16_rn(y[m] - __bfloat162float(hi));
        q16[warp * D + lane + 32 * m] = hi;
        q16[(G + warp) * D + lane + 32 * m] = lo;
      }
    }
    if (has_new && warp == 3) {
      float y[E];
      norm_rope(qkv_b + p.nq * D + h * D, p.k_norm, y);
      __nv_bfloat16* nk = reinterpret_cast<__nv_bfloat16*>(smem + CF::kOffNew);
      __nv_bfloat16* nv = nk + D;
      const float* vsrc = qkv_b + (p.nq + p.nkv) * D + h * D;
#pragma unroll
      for (int m = 0; m < E; ++m) {
        const int e = lane + 32 * m;
        const __nv_bfloat16 kk = __float2bfloat16_rn(y[m]);
        const __nv_bfloat16 vv = __float2bfloat16_rn(vsrc[e]);
        nk[e] = kk;
        nv[e] = vv;
        kbase[static_cast<size_t>(P) * D + e] = kk;
        vbase[static_cast<size_t>(P) * D + e] = vv;
      }
    }
    __syncthreads();

    // A fragments of Q (rows g: hi for g < G, lo for G <= g < 2G; rows g+8 zero)
    uint32_t qa[D / 16][2];
    {
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(smem + CF::kOffQ);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        qa[kk][0] = q32[(g * D + kk * 16 + 2 * t) / 2];
        qa[kk][1] = q32[(g * D + kk * 16 + 8 + 2 * t) / 2];
      }
    }

    const float scale_log2 = kLog2e * rsqrtf(static_cast<float>(D));
    for (int it = 0; it < ntiles; ++it) {
      {  // refill the stage consumed in the previous iteration
        const int nxt = it + S - 1;
        if (nxt < ntiles) {
          const int sn = nxt % S;
          const int pos0 = pos_begin + nxt * kAttnTile;
          load_tile<D>(sStages + sn * CF::kStageBytes, kbase, pos0, pos_end);
          load_tile<D>(sStages + sn * CF::kStageBytes + CF::kTileBytes, vbase, pos0, pos_end);
        }
        cp_async_commit();
      }
      cp_async_wait<S - 1>();  // tile `it` has landed
      __syncthreads();
      const int st = it % S;
      const int tile_pos0 = pos_begin + it * kAttnTile;
      if (has_new && P >= tile_pos0 && P < tile_pos0 + kAttnTile) {
        // the cache row at P was read before this step's append: use the fresh values
        const int r = P - tile_pos0;
        const uint4* nk = reinterpret_cast<const uint4*>(smem + CF::kOffNew);
        const uint4* nv = nk + D / 8;
        if (tid < D / 8) {
          unsigned char* stg = smem + CF::kOffStages + st * CF::kStageBytes;
          *reinterpret_cast<uint4*>(stg + swz<D>(r, tid)) = nk[tid];
          *reinterpret_cast<uint4*>(stg + CF::kTileBytes + swz<D>(r, tid)) = nv[tid];
        }
        __syncthreads();
      }

      const uint32_t tK = sStages + st * CF::kStageBytes, tV = tK + CF::kTileBytes;
      const int wrow = warp * 16;  // this warp's 16 positions within the tile

      // ---- S = Q K^T (16 query rows x 16 positions)
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int mi = lane >> 3, rr = lane & 7;
        const int row = wrow + (mi >> 1) * 8 + rr;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t bfr[4];
          ldmatrix_x4(bfr, tK + swz<D>(row, 2 * kk + (mi & 1)));
          mma_bf16_16816(sacc[0], qa[kk][0], 0u, qa[kk][1], 0u, bfr[0], bfr[1]);
          mma_bf16_16816(sacc[1], qa[kk][0], 0u, qa[kk][1], 0u, bfr[2], bfr[3]);
        }
      }
      // scores of row g at positions wrow + 8 n + 2 t + {0, 1}
      float sv[4] = {sacc[0][0], sacc[0][1], sacc[1][0], sacc[1][1]};
#pragma unroll
      for (int i = 0; i < 4; ++i) sv[i] += __shfl_xor_sync(0xffffffffu, sv[i], 4 * G);  // hi + lo rows
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int pos = tile_pos0 + wrow + (i >> 1) * 8 + 2 * t + (i & 1);
        sv[i] = pos < pos_end ? sv[i] * scale_log2 : -INFINITY;
      }
      float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float mref = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
      float pr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pr[i] = exp2f(sv[i] - mref);
      l_run = l_run * corr + (pr[0] + pr[1]) + (pr[2] + pr[3]);
      m_run = m_new;
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        o[j][0] *= corr;
        o[j][1] *= corr;
      }
      // A operand of P: row g = hi (g < G) or lo (G <= g < 2G) part of this row's probabilities
      uint32_t pa0 = 0u, pa2 = 0u;
      if (g < G) {
        pa0 = pack_bf16x2(pr[0], pr[1]);
        pa2 = pack_bf16x2(pr[2], pr[3]);
      } else if (g < 2 * G) {
        float lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) lo[i] = pr[i] - __bfloat162float(__float2bfloat16_rn(pr[i]));
        pa0 = pack_bf16x2(lo[0], lo[1]);
        pa2 = pack_bf16x2(lo[2], lo[3]);
      }
      // ---- O += P V
      {
        const int mi = lane >> 3, rr = lane & 7;
        const int row = wrow + (mi & 1) * 8 + rr;
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
          uint32_t bfr[4];
          ldmatrix_x4_trans(bfr, tV + swz<D>(row, 2 * jj + (mi >> 1)));
          mma_bf16_16816(o[2 * jj], pa0, 0u, pa2, 0u, bfr[0], bfr[1]);
          mma_bf16_16816(o[2 * jj + 1], pa0, 0u, pa2, 0u, bfr[2], bfr[3]);
        }
      }
      __syncthreads();  // this stage is refilled in the next iteration
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  griddep_launch_dependents();

  // ---- per-warp state -> this CTA's (m, l, acc) per head (rows g < G after adding the lo rows)
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
#pragma unroll
  for (int j = 0; j < D / 8; ++j) {
    o[j][0] += __shfl_xor_sync(0xffffffffu, o[j][0], 4 * G);
    o[j][1] += __shfl_xor_sync(0xffffffffu, o[j][1], 4 * G);
  }
  // warp partials in the (now idle) stage area: [4 warps][G] m, l, then [4][G][D] o
  float* mw = reinterpret_cast<float*>(smem + CF::kOffStages);
  float* lw = mw + 4 * G;
  float* ow = lw + 4 * G;
  if (g < G) {
    if (t == 0) {
      mw[warp * G + g] = m_run;
      lw[warp * G + g] = l_run;
    }
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      ow[(warp * G + g) * D + 8 * j + 2 * t] = o[j][0];
      ow[(warp * G + g) * D + 8 * j + 2 * t + 1] = o[j][1];
    }
  }
  __syncthreads();
  float* fw = misc;  // [4][G] warp weights
  if (tid < G) {
    float M = -INFINITY;
    for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * G + tid]);
    float L = 0.f;
    for (int w = 0; w < 4; ++w) {
      const float f = (M == -INFINITY) ? 0.f : exp2f(mw[w * G + tid] - M);
      fw[w * G + tid] = f;
      L += f * lw[w * G + tid];
    }
    xchg[tid * (D + 2)] = M;
    xchg[tid * (D + 2) + 1] = L;
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += kAttnThreads) {
    const int j = i / D, e = i % D;
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) a += fw[w * G + j] * ow[(w * G + j) * D + e];
    xchg[j * (D + 2) + 2 + e] = a;
  }

  // ---- cluster merge: CTA `rank` combines outputs [rank * n, (rank + 1) * n) of all C CTAs
  cluster_sync();
  {
    constexpr int kOut = G * D;
    constexpr int kPer = (kOut + C - 1) / C;
    const uint32_t xa = smem_u32(xchg);
    float* out_b = p.out + static_cast<size_t>(b) * p.nq * D + h * G * D;
    const int i_end = (rank + 1) * kPer < kOut ? (rank + 1) * kPer : kOut;
    for (int i = rank * kPer + tid; i < i_end; i += kAttnThreads) {
      const int j = i / D, e = i % D;
      float mr[C], lr[C], ar[C];
#pragma unroll
      for (int r = 0; r < C; ++r) {
        const uint32_t base = map_rank(xa, static_cast<uint32_t>(r));
        mr[r] = ld_cluster_f32(base + (j * (D + 2)) * 4);
        lr[r] = ld_cluster_f32(base + (j * (D + 2) + 1) * 4);
        ar[r] = ld_cluster_f32(base + (j * (D + 2) + 2 + e) * 4);
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < C; ++r) M = fmaxf(M, mr[r]);
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int r = 0; r < C; ++r) {
        const float f = (mr[r] == -INFINITY) ? 0.f : exp2f(mr[r] - M);
        num = fmaf(f, ar[r], num);
        den = fmaf(f, lr[r], den);
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
  }
  cluster_sync();  // no CTA leaves while others may still read its shared memory
  tl_mark(p.tl, 2);
}

namespace {

template <int D, int G>
cudaError_t launch_attn_t(const LaunchCtx& c, const AttnParams& p) {
  constexpr int C = kAttnCluster;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, p.nkv, p.B);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = AttnCfg<D>::kBytes;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_attention<D, G, C>, p);
}

template <int D, int G>
cudaError_t prepare_attn_t() {
  return cudaFuncSetAttribute(k_attention<D, G, kAttnCluster>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(AttnCfg<D>::kBytes));
}

}  // namespace

size_t attention_smem_bytes(int head_dim) {
  return head_dim == 64 ? AttnCfg<64>::kBytes : AttnCfg<128>::kBytes;
}

cudaError_t prepare_attention(int head_dim, int G) {
#define DEC_ATTN_PREP(D_, G_) \
  if (head_dim == D_ && G == G_) return prepare_attn_t<D_, G_>();
  DEC_ATTN_PREP(64, 1)
  DEC_ATTN_PREP(64, 2)
  DEC_ATTN_PREP(64, 4)
  DEC_ATTN_PREP(128, 1)
  DEC_ATTN_PREP(128, 2)
  DEC_ATTN_PREP(128, 4)
#undef DEC_ATTN_PREP
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention(const LaunchCtx& c, const AttnParams& p, int head_dim) {
  const int G = p.nq / p.nkv;
#define DEC_ATTN_CASE(D_, G_) \
  if (head_dim == D_ && G == G_) return launch_attn_t<D_, G_>(c, p);
  DEC_ATTN_CASE(64, 1)
  DEC_ATTN_CASE(64, 2)
  DEC_ATTN_CASE(64, 4)
  DEC_ATTN_CASE(128, 1)
  DEC_ATTN_CASE(128, 2)
  DEC_ATTN_CASE(128, 4)
#undef DEC_ATTN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dec

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
// Grid: (max_splits, n_kv, B).  A CTA takes split s of sequence b, KV head h:
// positions [s*L, min((s+1)*L, P+1)).  K/V tiles of 64 positions are staged in
// shared memory with cp.async (zero-filled past the split, XOR-swizzled 16-byte
// chunks so ldmatrix is conflict-free), double-buffered.  Each of the 4 warps
// takes 16 positions of a tile and runs the two products on tensor cores
// (mma.sync m16n8k16, bf16 in, fp32 accumulate): the GQA group's G query heads
// share every K/V row, so scores and the weighted sum are small dense products.
// Precision: q and the probabilities are split into bf16 hi + lo rows (rows
// 0..G-1 and G..2G-1 of the 16-row A operand), which keeps ~16 significant bits
// while K/V are bf16 already.  Softmax statistics are fp32 in the exp2 domain.
// The last CTA to finish a (b, h) merges the splits in split order.
#include "dec_internal.cuh"

namespace dec {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct AttnSmem {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = kAttnTile * kRowBytes;
  static constexpr int kQBytes = 16 * kRowBytes;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;          // 2 stages
  static constexpr int kOffV = kOffK + 2 * kTileBytes;   // 2 stages
  static constexpr int kOffNew = kOffV + 2 * kTileBytes; // new k row, new v row (bf16)
  static constexpr int kOffMisc = kOffNew + 2 * kRowBytes;
  static constexpr int kMiscFloats = 2048 + 16;          // merge factors and sums + per-head stats
  static constexpr int kBytes = kOffMisc + kMiscFloats * 4;
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

}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kAttnThreads) k_attention(AttnParams p) {
  using SM = AttnSmem<D>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ unsigned s_ticket;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  int P = p.positions[b];
  P = P < 0 ? 0 : (P >= p.max_ctx ? p.max_ctx - 1 : P);  // flagged by the embedding kernel
  const int T = P + 1;
  const int nsplit = (T + p.split_len - 1) / p.split_len;
  if (split >= nsplit) {
    griddep_launch_dependents();
    return;
  }
  const int pos_begin = split * p.split_len;
  const int pos_end = min(pos_begin + p.split_len, T);
  const int ntiles = (pos_end - pos_begin + kAttnTile - 1) / kAttnTile;
  const bool has_new = (P >= pos_begin && P < pos_end);

  const size_t plane = static_cast<size_t>(p.B) * p.nkv * p.max_ctx * D;
  const size_t head_off = (static_cast<size_t>(b) * p.nkv + h) * p.max_ctx * D;
  __nv_bfloat16* kbase = p.kv + (static_cast<size_t>(p.layer) * 2 + 0) * plane + head_off;
  __nv_bfloat16* vbase = p.kv + (static_cast<size_t>(p.layer) * 2 + 1) * plane + head_off;

  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + SM::kOffQ, sK = s_base + SM::kOffK, sV = s_base + SM::kOffV;
  float* misc = reinterpret_cast<float*>(smem + SM::kOffMisc);

  // Tile 0 of the cached K/V does not depend on upstream kernels of this step.
  load_tile<D>(sK, kbase, pos_begin, pos_end);
  load_tile<D>(sV, vbase, pos_begin, pos_end);
  cp_async_commit();

  // zero the unused rows of the Q operand
  {
    uint32_t* q32 = reinterpret_cast<uint32_t*>(smem + SM::kOffQ);
    for (int i = tid; i < 16 * D / 2; i += kAttnThreads) q32[i] = 0u;
  }

  griddep_wait();
  __syncthreads();

  // ---- q/k per-head RMSNorm + RoPE (+ KV append by the split holding slot P)
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
    __nv_bfloat16* q16 = reinterpret_cast<__nv_bfloat16*>(smem + SM::kOffQ);
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
    __nv_bfloat16* nk = reinterpret_cast<__nv_bfloat16*>(smem + SM::kOffNew);
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
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(smem + SM::kOffQ);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = q32[(g * D + kk * 16 + 2 * t) / 2];
      qa[kk][1] = q32[(g * D + kk * 16 + 8 + 2 * t) / 2];
    }
  }

  const float scale_log2 = kLog2e * rsqrtf(static_cast<float>(D));
  float m_run = -INFINITY, l_run = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  for (int it = 0; it < ntiles; ++it) {
    const int st = it & 1;
    const int tile_pos0 = pos_begin + it * kAttnTile;
    if (it + 1 < ntiles) {
      const int nst = st ^ 1;
      load_tile<D>(sK + nst * SM::kTileBytes, kbase, tile_pos0 + kAttnTile, pos_end);
      load_tile<D>(sV + nst * SM::kTileBytes, vbase, tile_pos0 + kAttnTile, pos_end);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (has_new && P >= tile_pos0 && P < tile_pos0 + kAttnTile) {
      // the cache row at P was read before this step's append: use the fresh values
      const int r = P - tile_pos0;
      const uint4* nk = reinterpret_cast<const uint4*>(smem + SM::kOffNew);
      const uint4* nv = nk + D / 8;
      if (tid < D / 8) {
        *reinterpret_cast<uint4*>(smem + SM::kOffK + st * SM::kTileBytes + swz<D>(r, tid)) = nk[tid];
        *reinterpret_cast<uint4*>(smem + SM::kOffV + st * SM::kTileBytes + swz<D>(r, tid)) = nv[tid];
      }
      __syncthreads();
    }

    const uint32_t tK = sK + st * SM::kTileBytes, tV = sV + st * SM::kTileBytes;
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
    __syncthreads();  // this stage is refilled two iterations later
  }
  griddep_launch_dependents();

  // ---- per-warp state -> CTA state (rows g < G hold head g after adding the lo row)
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
#pragma unroll
  for (int j = 0; j < D / 8; ++j) {
    o[j][0] += __shfl_xor_sync(0xffffffffu, o[j][0], 4 * G);
    o[j][1] += __shfl_xor_sync(0xffffffffu, o[j][1], 4 * G);
  }
  // merge area (reuses the K stages): [4 warps][G] m, l, then [4][G][D] o
  float* mw = reinterpret_cast<float*>(smem + SM::kOffK);
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
  // CTA-level (M, L) per head and scale factors per warp
  float* fw = misc;                // [4][G]
  float* cta_ml = misc + 4 * G;    // [G][2]
  if (tid < G) {
    float M = -INFINITY;
    for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * G + tid]);
    float L = 0.f;
    for (int w = 0; w < 4; ++w) {
      const float f = exp2f(mw[w * G + tid] - M);
      fw[w * G + tid] = f;
      L += f * lw[w * G + tid];
    }
    cta_ml[2 * tid] = M;
    cta_ml[2 * tid + 1] = L;
  }
  __syncthreads();

  const int qoff = h * G * D;  // first query head of this group, in elements of out[b]
  float* out_b = p.out + static_cast<size_t>(b) * p.nq * D;
  if (nsplit == 1) {
    for (int i = tid; i < G * D; i += kAttnThreads) {
      const int j = i / D, e = i % D;
      float a = 0.f;
      for (int w = 0; w < 4; ++w) a += fw[w * G + j] * ow[(w * G + j) * D + e];
      out_b[qoff + i] = a / cta_ml[2 * j + 1];
    }
    return;
  }

  const int rec = G * (D + 2);
  float* part = p.partials + ((static_cast<size_t>(b) * p.nkv + h) * p.max_splits) * rec;
  float* mine = part + static_cast<size_t>(split) * rec;
  for (int i = tid; i < G * D; i += kAttnThreads) {
    const int j = i / D, e = i % D;
    float a = 0.f;
    for (int w = 0; w < 4; ++w) a += fw[w * G + j] * ow[(w * G + j) * D + e];
    mine[j * (D + 2) + 2 + e] = a;
  }
  if (tid < G) {
    mine[tid * (D + 2)] = cta_ml[2 * tid];
    mine[tid * (D + 2) + 1] = cta_ml[2 * tid + 1];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_ticket = atomicAdd(&p.counters[b * p.nkv + h], 1u);
  __syncthreads();
  if (s_ticket != static_cast<unsigned>(nsplit - 1)) return;
  __threadfence();

  // ---- last CTA of (b, h): log-sum-exp merge of the nsplit partials in split order
  float* fac = misc;          // [nsplit][G]: first M_s, then e^(M_s - M)
  float* lsp = misc + 1024;   // [nsplit][G]: L_s
  float* tot = misc + 2048;   // [G] merged denominators
  for (int i = tid; i < nsplit * G; i += kAttnThreads) {
    const int s = i / G, j = i % G;
    const float* r = part + static_cast<size_t>(s) * rec + j * (D + 2);
    fac[i] = __ldcg(r);
    lsp[i] = __ldcg(r + 1);
  }
  __syncthreads();
  if (warp < G) {  // warp j reduces head j over the splits
    float M = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, fac[s * G + warp]);
    M = warp_max(M);
    float L = 0.f;
    for (int s = lane; s < nsplit; s += 32) {
      const float f = exp2f(fac[s * G + warp] - M);
      fac[s * G + warp] = f;
      L += f * lsp[s * G + warp];
    }
    L = warp_sum(L);
    if (lane == 0) tot[warp] = L;
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += kAttnThreads) {
    const int j = i / D, e = i % D;
    const float* src = part + j * (D + 2) + 2 + e;
    float a = 0.f;
#pragma unroll 8
    for (int s = 0; s < nsplit; ++s) a = fmaf(fac[s * G + j], __ldcg(src + static_cast<size_t>(s) * rec), a);
    out_b[qoff + i] = a / tot[j];
  }
  if (tid == 0) p.counters[b * p.nkv + h] = 0u;
}

void attention_split_plan(int batch, int n_kv, int group, int max_ctx, int num_sms, int* split_len,
                          int* max_splits) {
  // Splits of 64 * 2^k positions: the shortest length that keeps the grid at the
  // full context within two CTAs per SM, capped at 512 positions, and at most
  // 1024 / group splits so the merge factors fit in shared memory.
  int L = kAttnTile;
  auto ns = [&](int len) { return (max_ctx + len - 1) / len; };
  while (L < 512 && (static_cast<long long>(batch) * n_kv * ns(L) > 2ll * num_sms || ns(L) * group > 1024)) L *= 2;
  while (ns(L) * group > 1024) L *= 2;
  *split_len = L;
  *max_splits = ns(L);
}

size_t attention_partials_floats(int batch, int n_kv, int group, int head_dim, int max_splits) {
  return static_cast<size_t>(batch) * n_kv * max_splits * group * (head_dim + 2);
}

size_t attention_smem_bytes(int head_dim) {
  return head_dim == 64 ? AttnSmem<64>::kBytes : AttnSmem<128>::kBytes;
}

template <int D, int G>
static cudaError_t launch_attn_t(const LaunchCtx& c, const AttnParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.max_splits, p.nkv, p.B);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = AttnSmem<D>::kBytes;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_attention<D, G>, p);
}

template <int D, int G>
static cudaError_t prepare_attn_t() {
  return cudaFuncSetAttribute(k_attention<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(AttnSmem<D>::kBytes));
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

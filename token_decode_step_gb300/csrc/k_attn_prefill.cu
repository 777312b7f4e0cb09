// Causal attention of a prefill chunk: T new tokens per sequence attend, token t over the
// cache slots 0..P + t (P = the tokens cached before the chunk), after the chunk's own K/V
// were appended by k_kv_append.  Each K/V tile is staged once per CTA and serves all of the
// CTA's query rows, instead of one decode attention per row re-reading the sequence.
//
// Sources: oxinfer crate page, "Performance" (prefill is compute-bound: the prompt's tokens
// are processed together); ANEForge "LLMs on the ANE", introduction (prefill runs every
// prompt token through the model at once) and "Correctness" (q/k per-head RMSNorm before
// RoPE); Butter architecture.md, "SINGLE-TOKEN DECODE" (the per-layer order: rope, cache
// append, attention over the cache).
//
// Grid (query tiles, n_kv, sequences), 128 threads.  A CTA owns 64 query rows of one KV head:
// 64 / G tokens x the G query heads that share the head (row r = token r / G, head r % G), so
// every K/V row staged in shared memory is used by 64 rows.  Warp w computes rows 16 w ..
// 16 w + 15 with mma.sync m16n8k16 (bf16 in, fp32 accumulate): S = Q K^T over 64-position
// tiles, the causal mask per row, an online softmax in the exp2 domain, O += P V.  Q and the
// probabilities enter as bf16 hi + lo halves (two MMAs into one accumulator), ~16 significant
// bits, as in the decode attention.  K/V tiles arrive by 16-byte cp.async into XOR-swizzled
// rows through a two-stage ring; query tiles are issued last-first so the longest rows start
// first.
#include "dec_internal.cuh"

namespace dec {

namespace {

constexpr int kPfRows = 64;     // query rows per CTA
constexpr int kPfStages = 2;    // K/V tile ring
constexpr int kPfThreads = 128;

template <int D>
struct PfCfg {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kQBytes = kPfRows * kRowBytes;       // one plane of Q (hi or lo)
  static constexpr int kTileBytes = kAttnTile * kRowBytes;  // 64 positions
  static constexpr int kStageBytes = 2 * kTileBytes;        // K tile, then V tile
  static constexpr int kOffQhi = 0;
  static constexpr int kOffQlo = kQBytes;
  static constexpr int kOffStages = 2 * kQBytes;
  static constexpr int kBytes = kOffStages + kPfStages * kStageBytes;
};

// byte offset of 16-byte chunk c of row r in a tile of D-element bf16 rows
template <int D>
__device__ __forceinline__ int pf_swz(int r, int c) {
  return r * (D * 2) + ((c ^ (r & 7)) << 4);
}

template <int D>
__device__ __forceinline__ void pf_load_tile(uint32_t sdst, const __nv_bfloat16* plane_base, int pos0, int valid_end) {
  constexpr int kChunks = D / 8;
#pragma unroll
  for (int j = 0; j < kAttnTile * kChunks / kPfThreads; ++j) {
    const int idx = threadIdx.x + j * kPfThreads;
    const int r = idx / kChunks, c = idx % kChunks;
    const int pos = pos0 + r;
    const bool ok = pos < valid_end;
    cp_async16(sdst + pf_swz<D>(r, c), plane_base + static_cast<size_t>(ok ? pos : 0) * D + c * 8, ok ? 16 : 0);
  }
}

}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kPfThreads, 2) k_attn_prefill(AttnParams p) {
  using CF = PfCfg<D>;
  constexpr int kTok = kPfRows / G;  // tokens per CTA
  constexpr int E = D / 32;          // elements per lane in the row prologue
  extern __shared__ __align__(128) unsigned char smem[];

  tl_mark(p.tl, 0);
  const int T = p.T > 1 ? p.T : 1;
  const int qt = static_cast<int>(gridDim.x - 1 - blockIdx.x), h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int t0 = qt * kTok;
  const int t_last = (t0 + kTok < T ? t0 + kTok : T) - 1;
  int P = p.positions[b];
  P = P < 0 ? 0 : P;
  // last slot a row may read: position P + t, clamped like the embedding kernel (which flags it)
  auto limit = [&](int tok) {
    const int pos = P + (tok < T ? tok : T - 1);
    return pos < p.max_ctx ? pos : p.max_ctx - 1;
  };
  const int pos_end = limit(t_last) + 1;
  const int ntiles = (pos_end + kAttnTile - 1) / kAttnTile;

  const size_t plane = static_cast<size_t>(p.B / T) * p.nkv * p.max_ctx * D;
  const size_t head_off = (static_cast<size_t>(b) * p.nkv + h) * p.max_ctx * D;
  const __nv_bfloat16* kbase = p.kv + (static_cast<size_t>(p.layer) * 2 + 0) * plane + head_off;
  const __nv_bfloat16* vbase = p.kv + (static_cast<size_t>(p.layer) * 2 + 1) * plane + head_off;
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQhi = s_base + CF::kOffQhi, sQlo = s_base + CF::kOffQlo, sStages = s_base + CF::kOffStages;

  float wq[E];
#pragma unroll
  for (int m = 0; m < E; ++m) wq[m] = bf16_to_f(p.q_norm[lane + 32 * m]);

  griddep_wait();  // this chunk's K/V rows were appended by the previous kernel
  tl_mark(p.tl, 1);
#pragma unroll
  for (int s = 0; s < kPfStages - 1; ++s) {
    if (s < ntiles) {
      pf_load_tile<D>(sStages + s * CF::kStageBytes, kbase, s * kAttnTile, pos_end);
      pf_load_tile<D>(sStages + s * CF::kStageBytes + CF::kTileBytes, vbase, s * kAttnTile, pos_end);
    }
    cp_async_commit();
  }

  // ---- q rows: per-head RMSNorm, RoPE at the row's position, bf16 hi and lo planes
  {
    const int nqkv = (p.nq + 2 * p.nkv) * D;
    for (int r = warp; r < kPfRows; r += kPfThreads / 32) {
      const int tok = t0 + r / G, j = r % G;
      const int row = b * T + (tok < T ? tok : T - 1);
      const float* src = p.qkv + static_cast<size_t>(row) * nqkv + (h * G + j) * D;
      float x[E];
#pragma unroll
      for (int m = 0; m < E; ++m) x[m] = src[lane + 32 * m];
      float ss = 0.f;
#pragma unroll
      for (int m = 0; m < E; ++m) ss = fmaf(x[m], x[m], ss);
      ss = warp_sum(ss);
      const float inv = rsqrtf(ss / static_cast<float>(D) + p.eps);
#pragma unroll
      for (int m = 0; m < E; ++m) x[m] = (x[m] * inv) * wq[m];
      const float2* cs = p.rope + static_cast<size_t>(row) * (D / 2);
      float y[E];
#pragma unroll
      for (int m = 0; m < E / 2; ++m) {  // rotate-half pairs (e, e + D/2)
        const float2 c = cs[lane + 32 * m];
        const float a = x[m], z = x[m + E / 2];
        y[m] = a * c.x - z * c.y;
        y[m + E / 2] = z * c.x + a * c.y;
      }
#pragma unroll
      for (int m = 0; m < E; ++m) {
        const int e = lane + 32 * m;
        const __nv_bfloat16 hi = __float2bfloat16_rn(y[m]);
        const __nv_bfloat16 lo = __float2bfloat16_rn(y[m] - __bfloat162float(hi));
        const int off = pf_swz<D>(r, e >> 3) + (e & 7) * 2;
        *reinterpret_cast<__nv_bfloat16*>(smem + CF::kOffQhi + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(smem + CF::kOffQlo + off) = lo;
      }
    }
  }

  // this lane's two rows (g, g + 8 of the warp's 16) and their last readable slots
  const int wr0 = warp * 16;
  const int lim0 = limit(t0 + (wr0 + g) / G), lim1 = limit(t0 + (wr0 + g + 8) / G);
  const int warp_lim = limit(t0 + (wr0 + 15) / G);  // the warp's longest row
  const float scale_log2 = 1.4426950408889634f * rsqrtf(static_cast<float>(D));
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  const int mi = lane >> 3, rr = lane & 7;

  for (int it = 0; it < ntiles; ++it) {
    {
      const int nxt = it + kPfStages - 1;
      if (nxt < ntiles) {
        const uint32_t st = sStages + (nxt % kPfStages) * CF::kStageBytes;
        pf_load_tile<D>(st, kbase, nxt * kAttnTile, pos_end);
        pf_load_tile<D>(st + CF::kTileBytes, vbase, nxt * kAttnTile, pos_end);
      }
      cp_async_commit();
    }
    cp_async_wait<kPfStages - 1>();
    __syncthreads();  // tile `it` (and, the first time, the q planes) visible to every warp
    const int pos0 = it * kAttnTile;
    if (pos0 <= warp_lim) {  // else every row of this warp ends before the tile
      const uint32_t tK = sStages + (it % kPfStages) * CF::kStageBytes, tV = tK + CF::kTileBytes;
      // ---- S = Q K^T: 16 rows x 64 positions (8 n-blocks of 8)
      float sacc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t qh[4], ql[4];
        ldmatrix_x4(qh, sQhi + pf_swz<D>(wr0 + (lane & 15), 2 * kk + (lane >> 4)));
        ldmatrix_x4(ql, sQlo + pf_swz<D>(wr0 + (lane & 15), 2 * kk + (lane >> 4)));
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
          uint32_t kf[4];
          ldmatrix_x4(kf, tK + pf_swz<D>(16 * nb + (mi >> 1) * 8 + rr, 2 * kk + (mi & 1)));
          mma_bf16_16816(sacc[2 * nb], qh[0], qh[1], qh[2], qh[3], kf[0], kf[1]);
          mma_bf16_16816(sacc[2 * nb], ql[0], ql[1], ql[2], ql[3], kf[0], kf[1]);
          mma_bf16_16816(sacc[2 * nb + 1], qh[0], qh[1], qh[2], qh[3], kf[2], kf[3]);
          mma_bf16_16816(sacc[2 * nb + 1], ql[0], ql[1], ql[2], ql[3], kf[2], kf[3]);
        }
      }
      // ---- scale, causal mask, online softmax (rows g: elements 0, 1; rows g + 8: 2, 3)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int pos = pos0 + 8 * n + 2 * t4 + (i & 1);
          const float v = pos <= ((i & 2) ? lim1 : lim0) ? sacc[n][i] * scale_log2 : -INFINITY;
          sacc[n][i] = v;
        }
        mx0 = fmaxf(mx0, fmaxf(sacc[n][0], sacc[n][1]));
        mx1 = fmaxf(mx1, fmaxf(sacc[n][2], sacc[n][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      // a row's first tile always holds slot 0, so mn is finite after it; the guards keep
      // exp2 away from (-inf) - (-inf)
      const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
      const float c0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0), c1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        sacc[n][0] = exp2f(sacc[n][0] - ref0);
        sacc[n][1] = exp2f(sacc[n][1] - ref0);
        sacc[n][2] = exp2f(sacc[n][2] - ref1);
        sacc[n][3] = exp2f(sacc[n][3] - ref1);
        s0 += sacc[n][0] + sacc[n][1];
        s1 += sacc[n][2] + sacc[n][3];
      }
      l0 = l0 * c0 + s0;
      l1 = l1 * c1 + s1;
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        o[j][0] *= c0;
        o[j][1] *= c0;
        o[j][2] *= c1;
        o[j][3] *= c1;
      }
      // ---- O += P V: k-steps of 16 positions; the S accumulators are the A fragments
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const float* pa = sacc[2 * ks];
        const float* pb = sacc[2 * ks + 1];
        const uint32_t h0 = pack_bf16x2(pa[0], pa[1]), h1 = pack_bf16x2(pa[2], pa[3]);
        const uint32_t h2 = pack_bf16x2(pb[0], pb[1]), h3 = pack_bf16x2(pb[2], pb[3]);
        auto rest = [](float v) { return v - __bfloat162float(__float2bfloat16_rn(v)); };
        const uint32_t q0 = pack_bf16x2(rest(pa[0]), rest(pa[1])), q1 = pack_bf16x2(rest(pa[2]), rest(pa[3]));
        const uint32_t q2 = pack_bf16x2(rest(pb[0]), rest(pb[1])), q3 = pack_bf16x2(rest(pb[2]), rest(pb[3]));
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
          uint32_t vf[4];
          ldmatrix_x4_trans(vf, tV + pf_swz<D>(16 * ks + (mi & 1) * 8 + rr, 2 * jj + (mi >> 1)));
          mma_bf16_16816(o[2 * jj], h0, h1, h2, h3, vf[0], vf[1]);
          mma_bf16_16816(o[2 * jj], q0, q1, q2, q3, vf[0], vf[1]);
          mma_bf16_16816(o[2 * jj + 1], h0, h1, h2, h3, vf[2], vf[3]);
          mma_bf16_16816(o[2 * jj + 1], q0, q1, q2, q3, vf[2], vf[3]);
        }
      }
    }
    __syncthreads();  // the stage is refilled in the next iteration
  }
  cp_async_wait<0>();

  // ---- normalise and store rows g, g + 8: out[(b T + token)][(h G + j) D + d]
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const int nqd = p.nq * D;
  const size_t plane_hl = static_cast<size_t>(p.B) * nqd;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = wr0 + g + 8 * half, tok = t0 + r / G, j = r % G;
    if (tok >= T) continue;
    const float inv = half ? inv1 : inv0;
    const size_t base = static_cast<size_t>(b * T + tok) * nqd + (h * G + j) * D + 2 * t4;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const float v0 = o[n][2 * half] * inv, v1 = o[n][2 * half + 1] * inv;
      *reinterpret_cast<float2*>(p.out + base + 8 * n) = make_float2(v0, v1);
      if (p.out_hl) {
        const __nv_bfloat16 a = __float2bfloat16_rn(v0), c = __float2bfloat16_rn(v1);
        __nv_bfloat162 hi, lo;
        hi.x = a;
        hi.y = c;
        lo.x = __float2bfloat16_rn(v0 - __bfloat162float(a));
        lo.y = __float2bfloat16_rn(v1 - __bfloat162float(c));
        *reinterpret_cast<__nv_bfloat162*>(p.out_hl + base + 8 * n) = hi;
        *reinterpret_cast<__nv_bfloat162*>(p.out_hl + plane_hl + base + 8 * n) = lo;
      }
    }
  }
  griddep_launch_dependents();
  tl_mark(p.tl, 2);
}

namespace {

template <int D, int G>
cudaError_t pf_launch(const LaunchCtx& c, const AttnParams& p, bool prepare) {
  if (prepare)
    return cudaFuncSetAttribute(k_attn_prefill<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, PfCfg<D>::kBytes);
  const int T = p.T > 1 ? p.T : 1;
  constexpr int kTok = kPfRows / G;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((T + kTok - 1) / kTok, p.nkv, p.B / T);
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = PfCfg<D>::kBytes;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_attn_prefill<D, G>, p);
}

cudaError_t pf_dispatch(const LaunchCtx& c, const AttnParams& p, int head_dim, int G, bool prepare) {
  if (head_dim == 128) {
    if (G == 1) return pf_launch<128, 1>(c, p, prepare);
    if (G == 2) return pf_launch<128, 2>(c, p, prepare);
    if (G == 4) return pf_launch<128, 4>(c, p, prepare);
  } else if (head_dim == 64) {
    if (G == 1) return pf_launch<64, 1>(c, p, prepare);
    if (G == 2) return pf_launch<64, 2>(c, p, prepare);
    if (G == 4) return pf_launch<64, 4>(c, p, prepare);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int attn_prefill_min_tokens() { return 16; }

cudaError_t prepare_attn_prefill(int head_dim, int G) {
  return pf_dispatch(LaunchCtx{nullptr, false}, AttnParams{}, head_dim, G, true);
}

cudaError_t launch_attn_prefill(const LaunchCtx& c, const AttnParams& p, int head_dim) {
  return pf_dispatch(c, p, head_dim, p.nq / p.nkv, false);
}

}  // namespace dec

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
// runs (multiples of 16 positions, so ragged batches stay balanced), CTA r takes
// run r.  Each CTA streams its K/V tiles of 64 positions into shared memory with
// cp.async through a ring of S stages (XOR-swizzled 16-byte chunks so ldmatrix is
// conflict-free; the first S-1 tiles are requested before the grid-dependency
// wait, which for small batches is the whole run) and runs both products on
// tensor cores (mma.sync m16n8k16, bf16 in, fp32
// accumulate): the group's G query heads share every K/V row.  q and the
// probabilities enter as bf16 hi + lo rows (rows 0..G-1 and G..2G-1 of the
// 16-row A operand), ~16 significant bits; softmax statistics are fp32 in the
// exp2 domain.  The C partial results are merged through distributed shared
// memory: every CTA stores its share of CTA r's 1/C slice of the outputs into CTA r's
// shared memory, one cluster barrier, then CTA r combines the slice (no global
// partials, no atomics, no remote loads).
#include <mutex>

#include "attn_common.cuh"
#include "dec_internal.cuh"

namespace dec {

namespace {

using attn::kLog2e;

// Two shapes of the stage ring: shallow (about 100 KB, two CTAs per SM, for grids
// above the SM count; deeper rings measured slower there) and deep (about 200 KB, one
// CTA per SM, for grids that fit on the SMs at once: up to 5 or 11 tiles are in
// flight before the wait).
template <int D, bool DEEP>
struct AttnCfg {
  static constexpr int kStages = DEEP ? (D == 128 ? 6 : 12) : (D == 128 ? 3 : 4);
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = kAttnTile * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;                  // K tile then V tile
  static constexpr int kOffQ = 0;                                      // [16][D] bf16
  static constexpr int kOffStages = 16 * kRowBytes;
  static constexpr int kOffNew = kOffStages + kStages * kStageBytes;  // new k row, new v row
  // cluster merge receive area
  static constexpr int kXchgFloats = attn::Xchg<D>::kFloats;
  static constexpr int kOffXchg = kOffNew + 2 * kRowBytes;
  static constexpr int kOffMisc = kOffXchg + kXchgFloats * 4;          // [4][G] floats
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

}  // namespace

template <int D, int G, int C, bool DEEP>
__global__ void __launch_bounds__(kAttnThreads) k_attention(AttnParams p) {
  using CF = AttnCfg<D, DEEP>;
  constexpr int S = CF::kStages;
  extern __shared__ __align__(128) unsigned char smem[];

  tl_mark(p.tl, 0);
  const int h = blockIdx.y, b = blockIdx.z;
  const int rank = static_cast<int>(attn::cluster_ctarank());
  // The merge writes into the other CTAs' shared memory: first barrier phase, completed
  // before the first remote store, so every CTA of the cluster is known to be running.
  attn::cluster_arrive_relaxed();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  // row b is token b % tps of sequence b / tps (tps = 1: the one new token)
  const int tps = p.T > 1 ? p.T : 1, seq = b / tps;
  int P = p.positions[seq] + b % tps;
  P = P < 0 ? 0 : (P >= p.max_ctx ? p.max_ctx - 1 : P);  // flagged by the embedding kernel
  const int T = P + 1;
  int pos_begin, pos_end;
  attn::attention_run(T, C, rank, &pos_begin, &pos_end);
  const int ntiles = (pos_end - pos_begin + kAttnTile - 1) / kAttnTile;
  // one token: this kernel appends slot P itself (and patches the stale copy it read);
  // a verify step appended every row's slot in the previous kernel
  const bool has_new = tps == 1 && (P >= pos_begin && P < pos_end);

  const size_t plane = static_cast<size_t>(p.B / tps) * p.nkv * p.max_ctx * D;
  const size_t head_off = (static_cast<size_t>(seq) * p.nkv + h) * p.max_ctx * D;
  __nv_bfloat16* kbase = p.kv + (static_cast<size_t>(p.layer) * 2 + 0) * plane + head_off;
  __nv_bfloat16* vbase = p.kv + (static_cast<size_t>(p.layer) * 2 + 1) * plane + head_off;

  const uint32_t s_base = smem_u32(smem);
  const uint32_t sStages = s_base + CF::kOffStages;
  float* xchg = reinterpret_cast<float*>(smem + CF::kOffXchg);  // receive area of the cluster merge
  float* misc = reinterpret_cast<float*>(smem + CF::kOffMisc);

  // Cached K/V tiles do not depend on upstream kernels of a one-token step: request the
  // first S-1 before the grid-dependency wait (a verify step's are requested after it,
  // since the previous kernel appended this step's slots).
  auto first_tiles = [&]() {
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
      if (s < ntiles) {
        const int pos0 = pos_begin + s * kAttnTile;
        load_tile<D>(sStages + s * CF::kStageBytes, kbase, pos0, pos_end);
        load_tile<D>(sStages + s * CF::kStageBytes + CF::kTileBytes, vbase, pos0, pos_end);
      }
      cp_async_commit();
    }
  };
  if (tps == 1) first_tiles();
  {  // zero the Q operand (rows 2G..15 stay zero)
    uint32_t* q32 = reinterpret_cast<uint32_t*>(smem + CF::kOffQ);
    for (int i = tid; i < 16 * D / 2; i += kAttnThreads) q32[i] = 0u;
  }
  // Norm weights and this sequence's RoPE factors (written by the embedding kernel,
  // two or more launches upstream) do not depend on the previous kernel either.
  constexpr int E = D / 32;  // elements per lane: lane + 32 m
  float wq[E], wk[E];
  float2 cs[E / 2];
#pragma unroll
  for (int m = 0; m < E; ++m) {
    wq[m] = bf16_to_f(p.q_norm[lane + 32 * m]);
    wk[m] = bf16_to_f(p.k_norm[lane + 32 * m]);
  }
  {
    const float2* rope_b = p.rope + static_cast<size_t>(b) * (D / 2);
#pragma unroll
    for (int m = 0; m < E / 2; ++m) cs[m] = rope_b[lane + 32 * m];
  }

  griddep_wait();
  tl_mark(p.tl, 1);
  if (tps > 1) first_tiles();
  __syncthreads();

  float m_run = -INFINITY, l_run = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  if (ntiles > 0) {
    // ---- q/k per-head RMSNorm + RoPE (+ KV append by the CTA holding slot P)
    const int nqkv = (p.nq + 2 * p.nkv) * D;
    const float* qkv_b = p.qkv + static_cast<size_t>(b) * nqkv;
    // rows of this step's q (warps < G, one head each) and, in the CTA holding slot P,
    // the new k and v (warp kvw); all loads are issued before any arithmetic
    constexpr int kvw = G < 4 ? G : 3;
    const bool do_q = warp < G, do_kv = has_new && warp == kvw;
    float xq[E], xk[E], xv[E];
    if (do_q) {
      const float* src = qkv_b + (h * G + warp) * D;
#pragma unroll
      for (int m = 0; m < E; ++m) xq[m] = src[lane + 32 * m];
    }
    if (do_kv) {
      const float* ksrc = qkv_b + p.nq * D + h * D;
      const float* vsrc = qkv_b + (p.nq + p.nkv) * D + h * D;
#pragma unroll
      for (int m = 0; m < E; ++m) {
        xk[m] = ksrc[lane + 32 * m];
        xv[m] = vsrc[lane + 32 * m];
      }
    }
    auto norm_rope = [&](float (&x)[E], const float (&wn)[E], float (&y)[E]) {
      float ss = 0.f;
#pragma unroll
      for (int m = 0; m < E; ++m) ss = fmaf(x[m], x[m], ss);
      ss = warp_sum(ss);
      const float inv = rsqrtf(ss / static_cast<float>(D) + p.eps);
#pragma unroll
      for (int m = 0; m < E; ++m) x[m] = (x[m] * inv) * wn[m];
      // pairs (e, e + D/2): lane's elements m and m + E/2
#pragma unroll
      for (int m = 0; m < E / 2; ++m) {
        const float a = x[m], c = x[m + E / 2];
        y[m] = a * cs[m].x - c * cs[m].y;
        y[m + E / 2] = c * cs[m].x + a * cs[m].y;
      }
    };
    if (do_q) {
      float y[E];
      norm_rope(xq, wq, y);
      __nv_bfloat16* q16 = reinterpret_cast<__nv_bfloat16*>(smem + CF::kOffQ);
#pragma unroll
      for (int m = 0; m < E; ++m) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(y[m]);
        const __nv_bfloat16 lo = __float2bfloat16_rn(y[m] - __bfloat162float(hi));
        q16[warp * D + lane + 32 * m] = hi;
        q16[(G + warp) * D + lane + 32 * m] = lo;
      }
    }
    if (do_kv) {
      float y[E];
      norm_rope(xk, wk, y);
      __nv_bfloat16* nk = reinterpret_cast<__nv_bfloat16*>(smem + CF::kOffNew);
      __nv_bfloat16* nv = nk + D;
#pragma unroll
      for (int m = 0; m < E; ++m) {
        const int e = lane + 32 * m;
        const __nv_bfloat16 kk = __float2bfloat16_rn(y[m]);
        const __nv_bfloat16 vv = __float2bfloat16_rn(xv[m]);
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
  attn::merge_store<D, G, C>(p, mw, lw, ow, xchg, misc, rank, b, h, tid);
  // Dependents are released only now: when their CTAs start earlier, on the SMs this
  // kernel runs on, their weight loads crowd the load/store pipe and the merge above
  // measured several times slower.
  griddep_launch_dependents();
  tl_mark(p.tl, 2);
}

// Verify step: the K/V of every row (token t of sequence b) into slot positions[b] + t,
// before any row attends.  One warp per (row, KV head): per-head RMSNorm and RoPE of
// k as in the attention prologue, bf16 rounding of k and v.
template <int D>
__global__ void __launch_bounds__(32) k_kv_append(AttnParams p) {
  tl_mark(p.tl, 0);
  const int h = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
  const int tps = p.T > 1 ? p.T : 1, seq = b / tps;
  int P = p.positions[seq] + b % tps;
  P = P < 0 ? 0 : (P >= p.max_ctx ? p.max_ctx - 1 : P);  // flagged by the embedding kernel
  constexpr int E = D / 32;
  float wk[E];
  float2 cs[E / 2];
#pragma unroll
  for (int m = 0; m < E; ++m) wk[m] = bf16_to_f(p.k_norm[lane + 32 * m]);
#pragma unroll
  for (int m = 0; m < E / 2; ++m) cs[m] = p.rope[static_cast<size_t>(b) * (D / 2) + lane + 32 * m];
  griddep_wait();
  tl_mark(p.tl, 1);
  const float* qkv_b = p.qkv + static_cast<size_t>(b) * (p.nq + 2 * p.nkv) * D;
  float x[E], v[E];
#pragma unroll
  for (int m = 0; m < E; ++m) {
    x[m] = qkv_b[p.nq * D + h * D + lane + 32 * m];
    v[m] = qkv_b[(p.nq + p.nkv) * D + h * D + lane + 32 * m];
  }
  float ss = 0.f;
#pragma unroll
  for (int m = 0; m < E; ++m) ss = fmaf(x[m], x[m], ss);
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / static_cast<float>(D) + p.eps);
#pragma unroll
  for (int m = 0; m < E; ++m) x[m] = (x[m] * inv) * wk[m];
  const size_t plane = static_cast<size_t>(p.B / tps) * p.nkv * p.max_ctx * D;
  const size_t slot = ((static_cast<size_t>(seq) * p.nkv + h) * p.max_ctx + P) * D;
  __nv_bfloat16* kd = p.kv + static_cast<size_t>(p.layer) * 2 * plane + slot;
  __nv_bfloat16* vd = kd + plane;
#pragma unroll
  for (int m = 0; m < E / 2; ++m) {  // rotate-half pairs (e, e + D/2)
    const float a = x[m], c = x[m + E / 2];
    kd[lane + 32 * m] = __float2bfloat16_rn(a * cs[m].x - c * cs[m].y);
    kd[lane + 32 * (m + E / 2)] = __float2bfloat16_rn(c * cs[m].x + a * cs[m].y);
  }
#pragma unroll
  for (int m = 0; m < E; ++m) vd[lane + 32 * m] = __float2bfloat16_rn(v[m]);
  griddep_launch_dependents();
  tl_mark(p.tl, 2);
}

namespace {

template <int D, int G, int C, bool DEEP>
struct Bf16Kern {
  static constexpr size_t kSmem = AttnCfg<D, DEEP>::kBytes;
  static auto kernel() { return k_attention<D, G, C, DEEP>; }
};

// Per device, KV format, head_dim and group: SM count and co-resident clusters per
// shape, filled by prepare_attention (before any capture), read by launch_attention.
constexpr int kMaxAttnDevices = 64;
struct AttnCaps {
  int num_sms = 0;
  int max_clusters[attn::kShapes] = {0, 0, 0, 0, 0};
};
AttnCaps g_caps[kMaxAttnDevices][2][2][3];
std::mutex g_caps_mu;

int fmt_index(int kv_fmt) { return kv_fmt == DEC_KV_AFFINE8_G64 ? 1 : 0; }
int dim_index(int head_dim) { return head_dim == 64 ? 0 : 1; }
int group_index(int G) { return G == 1 ? 0 : G == 2 ? 1 : 2; }

}  // namespace

size_t attention_smem_bytes(int head_dim) {
  return head_dim == 64 ? AttnCfg<64, false>::kBytes : AttnCfg<128, false>::kBytes;
}

// The widest shape whose grid runs in one wave with one CTA per SM: 16-, then 12-, then
// 8-CTA clusters with the deep ring when B n_kv of them fit at once (the occupancy
// query counts what the GPCs can place); with two CTAs per SM, 8-CTA clusters while they
// make one wave, 4-CTA clusters beyond that.  In grids of several waves every CTA pays
// its prologue, first-tile latency and cluster merge once: 4-CTA clusters halve the
// number of CTAs and measured faster than 8 (and than 2) for both cache formats, while
// keeping ragged batches balanced.
int attention_shape(int B, int nkv, int head_dim, int G, int kv_fmt) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxAttnDevices) return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  if (G != 1 && G != 2 && G != 4) return 0;
  AttnCaps caps;
  {
    std::lock_guard<std::mutex> lock(g_caps_mu);
    caps = g_caps[dev][fmt_index(kv_fmt)][dim_index(head_dim)][group_index(G)];
  }
  const long long clusters = static_cast<long long>(B) * nkv;
  if (caps.num_sms <= 0) return 0;
  if (clusters * 16 <= caps.num_sms && clusters <= caps.max_clusters[2]) return 2;
  if (clusters * 12 <= caps.num_sms && clusters <= caps.max_clusters[3]) return 3;
  if (clusters * 8 <= caps.num_sms && clusters <= caps.max_clusters[1]) return 1;
  // two CTAs per SM: clusters of 4 once clusters of 8 take more than one wave
  if (clusters * 8 > 2ll * caps.num_sms && caps.max_clusters[4] > 0) return 4;
  return 0;
}

cudaError_t prepare_attention(int head_dim, int G, int kv_fmt) {
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  AttnCaps caps;
  caps.num_sms = sms;
  e = kv_fmt == DEC_KV_AFFINE8_G64 ? prepare_attention_q8(head_dim, G, caps.max_clusters)
                                   : attn::prepare_dims<Bf16Kern>(head_dim, G, caps.max_clusters);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxAttnDevices) {
    std::lock_guard<std::mutex> lock(g_caps_mu);
    g_caps[dev][fmt_index(kv_fmt)][dim_index(head_dim)][group_index(G)] = caps;
  }
  return cudaSuccess;
}

cudaError_t launch_kv_append(const LaunchCtx& c, const AttnParams& p, int head_dim) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nkv, p.B);
  cfg.blockDim = dim3(32);
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.kv_fmt == DEC_KV_AFFINE8_G64) return launch_kv_append_q8(cfg, p, head_dim);
  if (head_dim == 64) return cudaLaunchKernelEx(&cfg, k_kv_append<64>, p);
  if (head_dim == 128) return cudaLaunchKernelEx(&cfg, k_kv_append<128>, p);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention(const LaunchCtx& c, const AttnParams& p, int head_dim) {
  const int shape = attention_shape(p.B, p.nkv, head_dim, p.nq / p.nkv, p.kv_fmt);
  if (p.kv_fmt == DEC_KV_AFFINE8_G64) return launch_attention_q8(c, p, head_dim, shape);
  return attn::launch_dims<Bf16Kern>(c, p, head_dim, shape);
}

}  // namespace dec

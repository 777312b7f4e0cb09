// Decode attention over an affine 8-bit KV cache (a code per element, a bf16 scale and
// bias per 64 elements of a row), the append of new rows in that form, and the quantizer.
//
// Sources: Butter architecture.md, model-layer section (AffineQuantizedKVCache among the
// per-layer cache types) and figure "SINGLE-TOKEN DECODE" (rope at offset = cache length,
// cache.append, sdpa_decode over the cache); oxinfer crate page, "MLX checkpoints"
// (value = scale * q + bias, one bf16 scale and bias per group of 64); ANEForge "LLMs on
// the ANE", "Correctness" and "What's inside" (per-head q/k RMSNorm before rotate-half
// RoPE; KV heads shared by groups of query heads).
//
// The split is the bf16 kernel's (clusters of C CTAs per (sequence, KV head), runs of 16
// positions, a ring of 64-position stages requested ahead, the log-sum-exp merge through
// distributed shared memory); what differs is how a stage becomes tensor-core operands:
//  * Codes enter mma.sync m16n8k16 as the f16 values 1024 + c: one byte_perm writes two
//    code bytes under the high byte 0x64 (an f16 of exponent 10, whose low mantissa bits
//    count by one).  For K the offset folds into the bias: scale (1024 + c) + (bias - 1024
//    scale) = scale c + bias (each product sums 64 dimensions and starts from zero every
//    stage).  V's codes are centred first, c - 128 (one exact f16 subtraction for two), with
//    bias + 128 scale: its products accumulate over every position of the run, and an
//    accumulator carrying 1024 times the weights' sum lost precision in proportion to the
//    run length (a systematic 1e-5 at 6000 positions before, measured).
//  * K: ldmatrix over the position-major code rows (a 16-byte piece = 16 codes of one
//    position); each thread receives four consecutive codes of a position, which become
//    its two f16x2 B registers.  The query's dimensions are permuted within each 16 to
//    match (element 4u + j of a piece is k index 2u + (j & 1) + 8 (j >> 1)).
//  * V: ldmatrix.trans over the same rows, two code bytes read as one 16-bit element: a
//    thread receives two positions x two dimensions, and byte_perm splits them into the B
//    registers of the even and of the odd dimension.
//  * The 16 A rows are (group, hi/lo part, head): each head's query restricted to the 64
//    dimensions of a group, as f16 hi + lo, and for the second product the probabilities
//    times the group's V scale, so rows 0..7 of every product carry group 0 and rows 8..15
//    group 1; the per-position scales and biases apply after the products.
//  * The probabilities times V scales are pre-scaled by a per-warp power of two that keeps
//    them inside the f16 range; the accumulators are rescaled when it drops and the factor
//    is removed at the end.
#include <cuda_fp16.h>

#include "attn_common.cuh"
#include "dec_internal.cuh"

namespace dec {

namespace {

using attn::kLog2e;

// Two shapes: deep (one CTA per SM: 128-position stages, each warp two independent
// 16-position chunks per stage, a five-stage ring at head_dim 128) and shallow (three CTAs
// per SM, 12 warps to hide the latency of each warp's dependent chains: 64-position stages,
// one chunk per warp, a three-stage ring, at most 170 registers).
template <int D, bool DEEP>
struct Q8Cfg {
  static constexpr int NG = D / 64;                        // groups of 64 per row
  static constexpr int CH = DEEP ? 2 : 1;                  // 16-position chunks per warp and stage
  static constexpr int kWarpPos = 16 * CH;                 // positions per warp and stage
  static constexpr int kTile = 4 * kWarpPos;               // positions per stage
  static constexpr int kMinBlocks = DEEP ? 1 : 3;          // CTAs per SM the registers are sized for
  static constexpr int kStages = DEEP ? (D == 128 ? 5 : 10) : (D == 128 ? 3 : 6);
  static constexpr int kCodeTile = kTile * D;              // one plane's codes
  static constexpr int kParTile = kTile * NG * 4;          // one plane's (scale, bias) pairs
  static constexpr int kStageBytes = 2 * kCodeTile + 2 * kParTile;  // K codes, V codes, K pairs, V pairs
  static constexpr int kOffQ = 0;                          // [16][D] f16 A operand
  static constexpr int kOffStages = 16 * D * 2;
  static constexpr int kOffNew = kOffStages + kStages * kStageBytes;  // new row: K, V codes; K, V pairs
  static constexpr int kNewBytes = (2 * D + 2 * NG * 4 + 15) / 16 * 16;
  // per warp [32 positions][NG] float4, over the Q operand (in registers before the first stage)
  static constexpr int kOffWp = kOffQ;
  static_assert(4 * kWarpPos * NG * 16 <= kOffStages, "per-warp floats must fit the Q operand's space");
  static constexpr int kOffXchg = kOffNew + kNewBytes;
  static constexpr int kOffMisc = kOffXchg + attn::Xchg<D>::kFloats * 4;  // merge weights, query group sums
  static constexpr int kBytes = kOffMisc + 64 * 4;
};

// byte offset of 16-byte piece c of row r inside a code tile (conflict-free ldmatrix)
template <int D>
__device__ __forceinline__ int swz8(int r, int c) {
  if constexpr (D == 128) {
    return r * 128 + ((c ^ (r & 7)) << 4);
  } else {
    return r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
  }
}

// k index (within a 16-dimension piece) at which the query element of dimension 4u + j sits
__device__ __forceinline__ int q8_kperm(int dim16) {
  return 2 * (dim16 >> 2) + (dim16 & 1) + 8 * ((dim16 >> 1) & 1);
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }

// two f16 1024 + c (from byte_perm) -> c - 128, exact: the V products accumulate centred codes, so
// that the running sums stay near the signal instead of carrying 1024 times the weights' sum
__device__ __forceinline__ uint32_t centre_codes(uint32_t x) {
  __half2 v = *reinterpret_cast<__half2*>(&x);
  return h2_bits(__hsub2(v, __float2half2_rn(1152.f)));
}

// 2^e for an integer e in [-126, 127], exact
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// One group of 64 values held two per lane of a warp (elements lane and 32 + lane):
// min-max affine 8-bit quantization, every decision in float32 (IEEE subtraction and
// division, rint halves to even).  Returns the (scale, bias) bf16 pair as one word, the
// scale in the low half; the lane's two codes in *c0, *c1.
__device__ __forceinline__ uint32_t quantize_group64(float x0, float x1, unsigned* c0, unsigned* c1) {
  float mn = fminf(x0, x1), mx = fmaxf(x0, x1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const __nv_bfloat16 s16 = __float2bfloat16_rn(__fdiv_rn(__fsub_rn(mx, mn), 255.f));
  const __nv_bfloat16 b16 = __float2bfloat16_rn(mn);
  const float s = __bfloat162float(s16), bias = __bfloat162float(b16);
  auto code = [&](float x) -> unsigned {
    if (s == 0.f) return 0u;
    const float q = rintf(__fdiv_rn(__fsub_rn(x, bias), s));
    return static_cast<unsigned>(fminf(fmaxf(q, 0.f), 255.f));
  };
  *c0 = code(x0);
  *c1 = code(x1);
  return static_cast<uint32_t>(__bfloat16_as_ushort(s16)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b16)) << 16);
}

// Quantize the row a warp holds (element lane + 32 m in x[m]) and store it at codes[0..D),
// pairs[0..NG) (global or shared memory).
template <int D>
__device__ __forceinline__ void store_row_q8(const float (&x)[D / 32], unsigned char* codes, uint32_t* pairs,
                                             int lane) {
#pragma unroll
  for (int gr = 0; gr < D / 64; ++gr) {
    unsigned c0, c1;
    const uint32_t sb = quantize_group64(x[2 * gr], x[2 * gr + 1], &c0, &c1);
    codes[64 * gr + lane] = static_cast<unsigned char>(c0);
    codes[64 * gr + 32 + lane] = static_cast<unsigned char>(c1);
    if (lane == 0) pairs[gr] = sb;
  }
}

// One stage: K and V codes of positions pos0.. (kTile of them; zero past valid_end) into swizzled
// tiles, then their (scale, bias) pairs (zero past valid_end, so masked positions stay finite).
template <int D, bool DEEP>
__device__ __forceinline__ void load_tile_q8(uint32_t stage, const unsigned char* kc, const unsigned char* vc,
                                             const unsigned char* kp, const unsigned char* vp, int pos0,
                                             int valid_end) {
  using CF = Q8Cfg<D, DEEP>;
  constexpr int NG = CF::NG;
  constexpr int kPieces = D / 16;
  constexpr int kTotal = CF::kTile * kPieces;
#pragma unroll
  for (int j = 0; j < kTotal / kAttnThreads; ++j) {
    const int idx = threadIdx.x + j * kAttnThreads;
    const int r = idx / kPieces, c = idx % kPieces;
    const int pos = pos0 + r;
    const bool ok = pos < valid_end;
    const size_t off = static_cast<size_t>(ok ? pos : 0) * D + c * 16;
    cp_async16(stage + swz8<D>(r, c), kc + off, ok ? 16 : 0);
    cp_async16(stage + CF::kCodeTile + swz8<D>(r, c), vc + off, ok ? 16 : 0);
  }
  constexpr int kParPieces = CF::kParTile / 16;  // 16-byte pieces of 4 / NG positions
  constexpr int kPosPerPiece = 4 / NG;
  const int i = threadIdx.x;
  if (i < 2 * kParPieces) {
    const int plane = i / kParPieces, q = i % kParPieces;
    const int p0 = pos0 + q * kPosPerPiece;
    int n = valid_end - p0;
    n = n < 0 ? 0 : (n > kPosPerPiece ? kPosPerPiece : n);
    const unsigned char* src = (plane ? vp : kp) + static_cast<size_t>(n > 0 ? p0 : 0) * NG * 4;
    cp_async16(stage + 2 * CF::kCodeTile + plane * CF::kParTile + q * 16, src, n * NG * 4);
  }
}

}  // namespace

template <int D, int G, int C, bool DEEP>
__global__ void __launch_bounds__(kAttnThreads, Q8Cfg<D, DEEP>::kMinBlocks) k_attention_q8(AttnParams p) {
  using CF = Q8Cfg<D, DEEP>;
  constexpr int S = CF::kStages;
  constexpr int NG = CF::NG;
  constexpr int CH = CF::CH;
  constexpr int kTile = CF::kTile;
  extern __shared__ __align__(128) unsigned char smem[];

  tl_mark(p.tl, 0);
  const int h = blockIdx.y, b = blockIdx.z;
  const int rank = static_cast<int>(attn::cluster_ctarank());
  attn::cluster_arrive_relaxed();  // first phase: completed before the merge's remote stores
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  // row b is token b % tps of sequence b / tps (tps = 1: the one new token)
  const int tps = p.T > 1 ? p.T : 1, seq = b / tps;
  int P = p.positions[seq] + b % tps;
  P = P < 0 ? 0 : (P >= p.max_ctx ? p.max_ctx - 1 : P);  // flagged by the embedding kernel
  const int T = P + 1;
  int pos_begin, pos_end;
  attn::attention_run(T, C, rank, &pos_begin, &pos_end);
  const int ntiles = (pos_end - pos_begin + kTile - 1) / kTile;
  const bool has_new = tps == 1 && (P >= pos_begin && P < pos_end);

  // (layer, plane, sequence, head) rows of the codes and of the pairs
  const size_t heads = static_cast<size_t>(p.B / tps) * p.nkv;
  const size_t krow = static_cast<size_t>(p.layer) * 2 * heads + static_cast<size_t>(seq) * p.nkv + h;
  const size_t vrow = krow + heads;
  unsigned char* kc = p.q8_codes + krow * p.max_ctx * D;
  unsigned char* vc = p.q8_codes + vrow * p.max_ctx * D;
  unsigned char* kp = p.q8_params + krow * p.max_ctx * NG * 4;
  unsigned char* vp = p.q8_params + vrow * p.max_ctx * NG * 4;

  const uint32_t s_base = smem_u32(smem);
  const uint32_t sStages = s_base + CF::kOffStages;
  float* xchg = reinterpret_cast<float*>(smem + CF::kOffXchg);
  float* misc = reinterpret_cast<float*>(smem + CF::kOffMisc);
  float* qs_s = misc + 32;  // [G][NG]: sum over a group's dimensions of a head's query (hi + lo)
  unsigned char* new_codes = smem + CF::kOffNew;  // [2][D]: this step's K, V codes
  uint32_t* new_pairs = reinterpret_cast<uint32_t*>(new_codes + 2 * D);  // [2][NG]

  auto first_tiles = [&]() {
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
      if (s < ntiles)
        load_tile_q8<D, DEEP>(sStages + s * CF::kStageBytes, kc, vc, kp, vp, pos_begin + s * kTile, pos_end);
      cp_async_commit();
    }
  };
  // cached tiles do not depend on upstream kernels of a one-token step
  if (tps == 1) first_tiles();
  {  // zero the Q operand
    uint32_t* q32 = reinterpret_cast<uint32_t*>(smem + CF::kOffQ);
    for (int i = tid; i < 16 * D / 2; i += kAttnThreads) q32[i] = 0u;
  }
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
  // O^T accumulators, one m16n8 tile per 16 dimensions s: rows g / g + 8 = dimensions
  // 16 s + 2 g / 16 s + 2 g + 1, columns 2t, 2t + 1 = head-rows (hi rows 0..G-1, lo rows G..2G-1)
  float o[D / 16][4];
#pragma unroll
  for (int j = 0; j < D / 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float bacc[NG];  // sum over positions of p (bias - 1024 scale) of V, per group
#pragma unroll
  for (int gr = 0; gr < NG; ++gr) bacc[gr] = 0.f;
  int e_run = 100;  // prescale exponent of the probabilities times V scales (warp-uniform)

  if (ntiles > 0) {
    // ---- q/k per-head RMSNorm + RoPE (+ quantized KV append by the CTA holding slot P)
    const int nqkv = (p.nq + 2 * p.nkv) * D;
    const float* qkv_b = p.qkv + static_cast<size_t>(b) * nqkv;
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
      __half* q16 = reinterpret_cast<__half*>(smem + CF::kOffQ);
      float qsum[NG];
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) qsum[gr] = 0.f;
#pragma unroll
      for (int m = 0; m < E; ++m) {
        const int dim = lane + 32 * m, gr = m >> 1;
        const __half hi = __float2half_rn(y[m]);
        const __half lo = __float2half_rn(y[m] - __half2float(hi));
        qsum[gr] += __half2float(hi) + __half2float(lo);
        const int col = (dim & ~15) + q8_kperm(dim & 15);
        q16[(gr * 8 + warp) * D + col] = hi;      // row (group, hi, head)
        q16[(gr * 8 + G + warp) * D + col] = lo;  // row (group, lo, head)
      }
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) {
        const float s = warp_sum(qsum[gr]);
        if (lane == 0) qs_s[warp * NG + gr] = s;
      }
    }
    if (do_kv) {
      float y[E];
      norm_rope(xk, wk, y);
      store_row_q8<D>(y, new_codes, new_pairs, lane);
      store_row_q8<D>(xv, new_codes + D, new_pairs + NG, lane);
      __syncwarp();
      // the new row into the cache (slot P): codes as 16-byte pieces, then the pairs
      if (lane < D / 16) {
        reinterpret_cast<uint4*>(kc + static_cast<size_t>(P) * D)[lane] = reinterpret_cast<const uint4*>(new_codes)[lane];
        reinterpret_cast<uint4*>(vc + static_cast<size_t>(P) * D)[lane] =
            reinterpret_cast<const uint4*>(new_codes + D)[lane];
      }
      if (lane < NG) {
        reinterpret_cast<uint32_t*>(kp)[static_cast<size_t>(P) * NG + lane] = new_pairs[lane];
        reinterpret_cast<uint32_t*>(vp)[static_cast<size_t>(P) * NG + lane] = new_pairs[NG + lane];
      }
    }
    __syncthreads();

    // A fragments of Q: rows g (group 0) and g + 8 (group 1)
    uint32_t qa[D / 16][4];
    {
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(smem + CF::kOffQ);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        qa[kk][0] = q32[(g * D + kk * 16 + 2 * t) / 2];
        qa[kk][2] = q32[(g * D + kk * 16 + 8 + 2 * t) / 2];
        if constexpr (NG == 2) {
          qa[kk][1] = q32[((g + 8) * D + kk * 16 + 2 * t) / 2];
          qa[kk][3] = q32[((g + 8) * D + kk * 16 + 8 + 2 * t) / 2];
        } else {
          qa[kk][1] = qa[kk][3] = 0u;
        }
      }
    }
    float qsl[NG];  // this lane's head (rows g < 2G; others read a valid, unused entry)
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) qsl[gr] = qs_s[(g % G) * NG + gr];
    const bool lo_part = g >= G, live_row = g < 2 * G;

    const float scale_log2 = kLog2e * rsqrtf(static_cast<float>(D));
    for (int it = 0; it < ntiles; ++it) {
      {  // refill the stage consumed in the previous iteration
        const int nxt = it + S - 1;
        if (nxt < ntiles)
          load_tile_q8<D, DEEP>(sStages + (nxt % S) * CF::kStageBytes, kc, vc, kp, vp, pos_begin + nxt * kTile,
                          pos_end);
        cp_async_commit();
      }
      cp_async_wait<S - 1>();  // stage `it` has landed
      __syncthreads();
      const int st = it % S;
      const int tile_pos0 = pos_begin + it * kTile;
      unsigned char* stg = smem + CF::kOffStages + st * CF::kStageBytes;
      if (has_new && P >= tile_pos0 && P < tile_pos0 + kTile) {
        // the cache row at P was read before this step's append: use the fresh values
        const int r = P - tile_pos0;
        if (tid < D / 16) {
          *reinterpret_cast<uint4*>(stg + swz8<D>(r, tid)) = reinterpret_cast<const uint4*>(new_codes)[tid];
          *reinterpret_cast<uint4*>(stg + CF::kCodeTile + swz8<D>(r, tid)) =
              reinterpret_cast<const uint4*>(new_codes + D)[tid];
        }
        if (tid < NG) {
          reinterpret_cast<uint32_t*>(stg + 2 * CF::kCodeTile)[r * NG + tid] = new_pairs[tid];
          reinterpret_cast<uint32_t*>(stg + 2 * CF::kCodeTile + CF::kParTile)[r * NG + tid] = new_pairs[NG + tid];
        }
        __syncthreads();
      }
      const int wrow = warp * CF::kWarpPos;  // this warp's CH chunks of 16 positions within the stage
      if (tile_pos0 + wrow < pos_end) {  // (warp-uniform: a stage's tail beyond the run is skipped)
        // ---- (scale, bias - 1024 scale) of K and V as floats for this warp's positions, and the prescale
        float4* wp = reinterpret_cast<float4*>(smem + CF::kOffWp) + warp * CF::kWarpPos * NG;
        float sv_max = 0.f;
        {  // pair q = (position q / NG, group q % NG) of this warp's positions
          const uint32_t* pkk = reinterpret_cast<const uint32_t*>(stg + 2 * CF::kCodeTile) + wrow * NG;
          const uint32_t* pvv = reinterpret_cast<const uint32_t*>(stg + 2 * CF::kCodeTile + CF::kParTile) + wrow * NG;
#pragma unroll
          for (int q = lane; q < CF::kWarpPos * NG; q += 32) {
            const uint32_t pk = pkk[q], pv = pvv[q];
            const float sk = __uint_as_float(pk << 16), bk = __uint_as_float(pk & 0xffff0000u);
            const float sv = __uint_as_float(pv << 16), bv = __uint_as_float(pv & 0xffff0000u);
            wp[q] = make_float4(sk, fmaf(-1024.f, sk, bk), sv, fmaf(128.f, sv, bv));
            sv_max = fmaxf(sv_max, fabsf(sv));
          }
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) sv_max = fmaxf(sv_max, __shfl_xor_sync(0xffffffffu, sv_max, o2));
        __syncwarp();
        // |p scale_V| 2^e < 2^14 for p <= 1: e = 13 - floor(log2 max|scale_V|)
        int e_tile = 100;
        if (sv_max > 0.f) {
          const int ex = static_cast<int>((__float_as_uint(sv_max) >> 23) & 0xffu) - 127;
          e_tile = 13 - ex < 100 ? 13 - ex : 100;
          e_tile = e_tile > -100 ? e_tile : -100;
        }
        int de = 0;
        if (e_tile < e_run) {
          de = e_tile - e_run;
          e_run = e_tile;
        }
        const float f_e = pow2i(e_run);
        const float f_de = de < -126 ? 0.f : pow2i(de);

        const uint32_t tK = sStages + st * CF::kStageBytes, tV = tK + CF::kCodeTile;

        // ---- S = Q K^T for both chunks: rows g (group 0) / g + 8 (group 1) x 16 positions each
        float sacc[CH][2][4];
#pragma unroll
        for (int c = 0; c < CH; ++c)
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) sacc[c][blk][0] = sacc[c][blk][1] = sacc[c][blk][2] = sacc[c][blk][3] = 0.f;
        {
          const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
          for (int kk = 0; kk < D / 16; kk += 2) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
              // matrices (block 0, piece), (0, piece + 1), (1, piece), (1, piece + 1) of chunk c
              const int row = wrow + 16 * c + (mi >> 1) * 8 + rr;
              uint32_t r4[4];
              ldmatrix_x4(r4, tK + swz8<D>(row, kk + (mi & 1)));
#pragma unroll
              for (int u = 0; u < 2; ++u) {
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                  const uint32_t w = r4[blk * 2 + u];
                  mma_f16_16816(sacc[c][blk], qa[kk + u][0], qa[kk + u][1], qa[kk + u][2], qa[kk + u][3],
                                __byte_perm(w, 0x64646464u, 0x4140), __byte_perm(w, 0x64646464u, 0x4342));
                }
              }
            }
          }
        }
        // scores of head (g % G) at positions wrow + 16 c + 8 blk + 2 t + i, with the V factors
        float sv[4 * CH], vs[4 * CH][NG], vb[4 * CH][NG];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int idx = c * 4 + blk * 2 + i, pl = 16 * c + 8 * blk + 2 * t + i;
              float sc = 0.f;
#pragma unroll
              for (int gr = 0; gr < NG; ++gr) {
                float s2 = sacc[c][blk][2 * gr + i];
                s2 += __shfl_xor_sync(0xffffffffu, s2, 4 * G);  // hi + lo rows
                const float4 f = wp[pl * NG + gr];
                sc = fmaf(f.x, s2, fmaf(f.y, qsl[gr], sc));
                vs[idx][gr] = f.z;
                vb[idx][gr] = f.w;
              }
              const int pos = tile_pos0 + wrow + pl;
              sv[idx] = pos < pos_end ? sc * scale_log2 : -INFINITY;
            }
          }
        }
        float mx = sv[0];
#pragma unroll
        for (int i = 1; i < 4 * CH; ++i) mx = fmaxf(mx, sv[i]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float mref = (m_new == -INFINITY) ? 0.f : m_new;
        const float corr = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
        float pr[4 * CH];
#pragma unroll
        for (int i = 0; i < 4 * CH; ++i) pr[i] = exp2f(sv[i] - mref);
        float psum = (pr[0] + pr[1]) + (pr[2] + pr[3]);
        if constexpr (CH == 2) psum += (pr[4] + pr[5]) + (pr[6] + pr[7]);
        l_run = l_run * corr + psum;
        m_run = m_new;
        if (!__all_sync(0xffffffffu, corr * f_de == 1.f)) {
          // this lane's accumulator columns are head-rows 2t and 2t + 1, whose factors the
          // lanes of those rows hold
          const float ca = __shfl_sync(0xffffffffu, corr, 8 * t) * f_de;
          const float cb = __shfl_sync(0xffffffffu, corr, 8 * t + 4) * f_de;
#pragma unroll
          for (int j = 0; j < D / 16; ++j) {
            o[j][0] *= ca;
            o[j][1] *= cb;
            o[j][2] *= ca;
            o[j][3] *= cb;
          }
        }
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) {
          bacc[gr] *= corr;
#pragma unroll
          for (int i = 0; i < 4 * CH; ++i) bacc[gr] = fmaf(pr[i], vb[i][gr], bacc[gr]);
        }
        // B operands of P^T per chunk and group: (k, column g) = head-row g at positions 2t..
        // (pa[c][gr], block 0) and 2t + 8.. (pa[c][2 + gr], block 1); hi rows the f16 value of
        // p scale_V 2^e, lo rows its remainder
        uint32_t pa[CH][4];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
            for (int gr = 0; gr < 2; ++gr) {
              uint32_t reg = 0u;
              if (gr < NG) {
                const int i0 = c * 4 + blk * 2;
                const float w0 = pr[i0] * f_e * vs[i0][gr < NG ? gr : 0];
                const float w1 = pr[i0 + 1] * f_e * vs[i0 + 1][gr < NG ? gr : 0];
                const __half2 hi = __floats2half2_rn(w0, w1);
                if (lo_part) {
                  const float2 hf = __half22float2(hi);
                  reg = h2_bits(__floats2half2_rn(w0 - hf.x, w1 - hf.y));
                } else {
                  reg = h2_bits(hi);
                }
                if (!live_row) reg = 0u;
              }
              pa[c][blk * 2 + gr] = reg;
            }
          }
        }
        // ---- O^T += V^T P^T: per chunk and 16-dimension piece s, A = the piece's codes (rows: its
        // even dimensions, then its odd ones; k = the chunk's 16 positions), B = that group's P^T
        {
          const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            // matrices (pos 0-7, piece), (8-15, piece), (0-7, piece + 1), (8-15, piece + 1) of chunk c
            const int row = wrow + 16 * c + (mi & 1) * 8 + rr;
#pragma unroll
            for (int jj = 0; jj < D / 16; jj += 2) {
              uint32_t r4[4];
              ldmatrix_x4_trans(r4, tV + swz8<D>(row, jj + (mi >> 1)));
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const uint32_t lo8 = r4[2 * u], hi8 = r4[2 * u + 1];
                const int sj = jj + u, gr = (NG == 2 && sj >= D / 32) ? 1 : 0;
                mma_f16_16816(o[sj], centre_codes(__byte_perm(lo8, 0x64646464u, 0x4240)),
                              centre_codes(__byte_perm(lo8, 0x64646464u, 0x4341)),
                              centre_codes(__byte_perm(hi8, 0x64646464u, 0x4240)),
                              centre_codes(__byte_perm(hi8, 0x64646464u, 0x4341)), pa[c][gr], pa[c][2 + gr]);
              }
            }
          }
        }
      }
      __syncthreads();  // this stage is refilled in the next iteration
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- per-warp state -> (m, l, o) per head in shared memory (lanes g < G)
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
#pragma unroll
  for (int gr = 0; gr < NG; ++gr) {
    bacc[gr] += __shfl_xor_sync(0xffffffffu, bacc[gr], 1);
    bacc[gr] += __shfl_xor_sync(0xffffffffu, bacc[gr], 2);
  }
  const float inv_e = pow2i(-e_run);
  float* mw = reinterpret_cast<float*>(smem + CF::kOffStages);
  float* lw = mw + 4 * G;
  float* ow = lw + 4 * G;
  {
    // head-rows 2t, 2t + 1 of this lane: add the lo rows (head-row + G), undo the prescale,
    // add the bias part of the head's group (held by the lanes of row = head)
    const int h0 = 2 * t, h1 = 2 * t + 1;
    float ba[2][NG];
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) {
      ba[0][gr] = __shfl_sync(0xffffffffu, bacc[gr], 4 * (h0 % G));
      ba[1][gr] = __shfl_sync(0xffffffffu, bacc[gr], 4 * (h1 % G));
    }
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      const int gr = (NG == 2 && j >= D / 32) ? 1 : 0;
      float v[4] = {o[j][0], o[j][1], o[j][2], o[j][3]};
      if constexpr (G == 1) {  // head-row 0 (hi) and 1 (lo) are this lane's two columns
        v[0] += v[1];
        v[2] += v[3];
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] += __shfl_xor_sync(0xffffffffu, v[q], G / 2);
      }
      const int dim = 16 * j + 2 * g;
      if (G == 1 ? t == 0 : h1 < G) {
        ow[(warp * G + h0) * D + dim] = fmaf(v[0], inv_e, ba[0][gr]);
        ow[(warp * G + h0) * D + dim + 1] = fmaf(v[2], inv_e, ba[0][gr]);
        if (G > 1) {
          ow[(warp * G + h1) * D + dim] = fmaf(v[1], inv_e, ba[1][gr]);
          ow[(warp * G + h1) * D + dim + 1] = fmaf(v[3], inv_e, ba[1][gr]);
        }
      }
    }
  }
  if (g < G && t == 0) {
    mw[warp * G + g] = m_run;
    lw[warp * G + g] = l_run;
  }
  __syncthreads();
  attn::merge_store<D, G, C>(p, mw, lw, ow, xchg, misc, rank, b, h, tid);
  // dependents are released only now (as in the bf16 kernel)
  griddep_launch_dependents();
  tl_mark(p.tl, 2);
}

// Verify step: the K/V of every row (token t of sequence b) into slot positions[b] + t, in
// the affine 8-bit form, before any row attends.  One warp per (row, KV head).
template <int D>
__global__ void __launch_bounds__(32) k_kv_append_q8(AttnParams p) {
  tl_mark(p.tl, 0);
  constexpr int NG = D / 64;
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
  float x[E], v[E], y[E];
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
#pragma unroll
  for (int m = 0; m < E / 2; ++m) {  // rotate-half pairs (e, e + D/2)
    const float a = x[m], c = x[m + E / 2];
    y[m] = a * cs[m].x - c * cs[m].y;
    y[m + E / 2] = c * cs[m].x + a * cs[m].y;
  }
  const size_t heads = static_cast<size_t>(p.B / tps) * p.nkv;
  const size_t krow = static_cast<size_t>(p.layer) * 2 * heads + static_cast<size_t>(seq) * p.nkv + h;
  const size_t vrow = krow + heads;
  store_row_q8<D>(y, p.q8_codes + (krow * p.max_ctx + P) * D,
                  reinterpret_cast<uint32_t*>(p.q8_params) + (krow * p.max_ctx + P) * NG, lane);
  store_row_q8<D>(v, p.q8_codes + (vrow * p.max_ctx + P) * D,
                  reinterpret_cast<uint32_t*>(p.q8_params) + (vrow * p.max_ctx + P) * NG, lane);
  griddep_launch_dependents();
  tl_mark(p.tl, 2);
}

// dec_kv_quantize: one warp per row of D floats.
template <int D>
__global__ void __launch_bounds__(128) k_kv_quantize(const float* __restrict__ src, int rows,
                                                     unsigned char* __restrict__ codes, uint32_t* __restrict__ pairs) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= rows) return;  // whole warps leave together
  float x[D / 32];
#pragma unroll
  for (int m = 0; m < D / 32; ++m) x[m] = src[static_cast<size_t>(row) * D + lane + 32 * m];
  store_row_q8<D>(x, codes + static_cast<size_t>(row) * D, pairs + static_cast<size_t>(row) * (D / 64), lane);
}

namespace {

template <int D, int G, int C, bool DEEP>
struct Q8Kern {
  static constexpr size_t kSmem = Q8Cfg<D, DEEP>::kBytes;
  static auto kernel() { return k_attention_q8<D, G, C, DEEP>; }
};

}  // namespace

cudaError_t prepare_attention_q8(int head_dim, int G, int (&max_clusters)[5]) {
  return attn::prepare_dims<Q8Kern>(head_dim, G, max_clusters);
}

cudaError_t launch_attention_q8(const LaunchCtx& c, const AttnParams& p, int head_dim, int shape) {
  return attn::launch_dims<Q8Kern>(c, p, head_dim, shape);
}

cudaError_t launch_kv_append_q8(const cudaLaunchConfig_t& cfg, const AttnParams& p, int head_dim) {
  if (head_dim == 64) return cudaLaunchKernelEx(&cfg, k_kv_append_q8<64>, p);
  if (head_dim == 128) return cudaLaunchKernelEx(&cfg, k_kv_append_q8<128>, p);
  return cudaErrorInvalidValue;
}

cudaError_t launch_kv_quantize(cudaStream_t s, const float* src, int rows, int head_dim, unsigned char* codes,
                               __nv_bfloat16* params) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid((rows + 3) / 4);
  uint32_t* pairs = reinterpret_cast<uint32_t*>(params);
  if (head_dim == 64) {
    k_kv_quantize<64><<<grid, 128, 0, s>>>(src, rows, codes, pairs);
  } else if (head_dim == 128) {
    k_kv_quantize<128><<<grid, 128, 0, s>>>(src, rows, codes, pairs);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace dec

// Internal declarations shared by the kernels and the C-ABI layer.
// Target: sm_103a (GB300).  No host-side torch types anywhere.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/dec.h"

namespace dec {

// ---------------------------------------------------------------- constants

constexpr int kResGroup = 8;        // rows per partial sum-of-squares of the residual
constexpr int kGemvRows = 8;        // rows per CTA of the batch-1 GEMV
constexpr int kAttnTile = 64;       // positions per attention smem tile
constexpr int kAttnThreads = 128;   // 4 warps, 16 positions each per tile
constexpr int kMaxTokensPerSeq = 4096;  // verify step / prefill chunk: new tokens per sequence
constexpr int kMaxRows = 65535;         // tokens per step (batch x tokens per sequence): a grid dimension
constexpr int kGroup = 64;          // affine 4-bit group size
constexpr int kGemmPrefetch = 4;    // 64-input weight units in flight per lane (batched path)

enum StatusBits : unsigned { kStatusBadToken = 1u, kStatusBadPos = 2u, kStatusTimeout = 4u };

enum Epilogue : int { kEpiStore = 0, kEpiResid = 1, kEpiSwiglu = 2, kEpiLmHead = 3 };
enum InMode : int { kInPlain = 0, kInNorm = 1 };
enum WFmt : int { kWBf16 = 0, kWQ4 = 1 };

// ---------------------------------------------------------------- kernel params

// Test hook: %globaltimer stamps of one launch in buf[3 idx ..]: 0 = first CTA start
// (atomic min), 1 = first CTA past the grid-dependency wait (min), 2 = last CTA end (max).
struct Timeline {
  unsigned long long* buf;
  int idx;
};

// Batch-1 GEMV: y = W x over a row tile (kGemvRows rows) and one K split.
struct GemvParams {
  Timeline tl;
  const void* w;            // bf16 [N][K] or q4 words uint32 [N][K/8]
  const uint32_t* sb;       // q4: scale (low 16 bits) | bias (high 16 bits), [N][K/64]
  int N, K, S, KS;          // rows, inputs, K splits, inputs per split
  // input vector (fp32 [K]); kInNorm: x = h * rsqrt(sum(sumsq_in)/K + eps) * norm_w
  const float* x;
  const __nv_bfloat16* norm_w;
  const float* sumsq_in;    // [n_sumsq_in]
  int n_sumsq_in;
  float eps;
  // epilogue
  float* out;               // store: y[N]; resid: h[N] (+=); swiglu: g[N/2]; lmhead: logits[N] or null
  float* sumsq_out;         // resid: [N / kResGroup]
  float* partials;          // [S][N] when S > 1
  unsigned* counters;       // [N / kGemvRows] (+1 for lmhead) zero on entry, left zero
  unsigned long long* amax_key;  // lmhead: packed (ordered value, ~index)
  int32_t* argmax_out;      // lmhead
  // Optional L2 prefetch of the cached K/V rows (positions 0..P-1) that the next
  // attention kernel reads: the CTAs split them into contiguous byte ranges.
  const unsigned char* pf_kv;     // this layer's K plane, V plane at + pf_plane_bytes; null: off
  const int32_t* pf_positions;    // [pf_B] cached positions P per sequence
  unsigned long long pf_plane_bytes, pf_head_bytes;  // one plane of a layer; one (sequence, head) run
  int pf_B, pf_nkv, pf_row_bytes, pf_max_ctx;
};

// Batched (B >= 2) projection on tensor cores over fragment-packed weight tiles.
struct GemmParams {
  Timeline tl;
  const void* w;            // packed tiles (see k_gemm_tc.cu)
  int N, Npad, K, S, KS, KC, B;  // rows, rows padded to 16, inputs, K splits, inputs per split,
                                 // inputs staged at once (divides KS), tokens
  int tblocks;              // token blocks of gemm_tc_block_tokens() tokens (1: all B tokens at once; > 1: S = 1)
  const __nv_bfloat16* xhl; // input as bf16 hi, lo planes [2][B][K] (norm inputs already times the norm weight)
  const float* sumsq_in;    // norm inputs: [B][n_sumsq_in] partial sums of squares of the residual
  int n_sumsq_in;
  float eps;
  float* out;               // store: [B][N]; resid: h [B][N] (+=); swiglu: g [B][N/2]; lmhead: logits [B][N] or null
  float* sumsq_out;         // resid: [B][N / kResGroup]
  __nv_bfloat16* xhl_out;   // resid: h * next_norm_w, swiglu: g, as hi, lo planes (the next consumer's input)
  const __nv_bfloat16* next_norm_w;  // resid: [N]
  float* partials;          // [S][Npad/16][32][NY*4] when S > 1
  unsigned* counters;       // [row blocks + 1], zero on entry, left zero
  unsigned long long* amax_key;  // lmhead: [B]
  int32_t* argmax_out;      // lmhead: [B]
};

// Prefill projections on tcgen05 (k_gemm_umma.cu): Y[M][N] = X[M][K] W[N][K]^T, X as bf16 hi, lo
// planes [2][M][K] and W bf16 [N][K] row-major, both read through TMA tensor maps.
struct UmmaParams {
  int M, N, K, m_tiles;     // tokens, weight rows, inputs (multiple of 64), ceil(M / 128)
  int tile_n;               // weight rows per tile: 128 or 256 (the weight map's box rows)
  int persistent;           // > 0: the persistent warp-specialized kernel on this many CTAs (one per SM)
  const float* sumsq_in;    // norm inputs: [M][n_sumsq_in] partial sums of squares of the residual
  int n_sumsq_in;
  float eps;
  float* out;               // store / lmhead: [M][N] (lmhead: may be null); resid: h [M][N] (+=); swiglu: g [M][N/2]
  float* sumsq_out;         // resid: [M][N / kResGroup]
  __nv_bfloat16* xhl_out;   // resid: h * next_norm_w, swiglu: g, as hi, lo planes
  const __nv_bfloat16* next_norm_w;  // resid: [N]
  unsigned long long* amax_key;      // lmhead: [M]
  int32_t* argmax_out;               // lmhead: [M]
  unsigned* counters;                // lmhead: one counter, zero on entry, left zero
  unsigned* status;                  // time-out flag (may be null)
};

// Batched decode projections of 4-bit weights on tcgen05 (k_gemm_q4tc.cu): Y[M][N] = X W^T for
// M <= 32 token rows; X as bf16 hi, lo planes [2][M][K] read through a TMA tensor map (boxes of
// 32 rows), W as row-major codes [N][K/2] bytes (a TMA tensor map) and sb words [N][K/64].
struct Q4tcParams {
  Timeline tl;
  int M, N, K, S;           // tokens (<= 32), weight rows, inputs (multiple of 64), K splits (dividing K / 64)
  int ctas;                 // persistent CTAs (one per SM)
  const uint32_t* sb;       // (scale | bias << 16) [N][K/64]
  const float* sumsq_in;    // norm inputs: [M][n_sumsq_in] partial sums of squares of the residual
  int n_sumsq_in;
  float eps;
  float* out;               // store / lmhead: [M][N] (lmhead: may be null); resid: h [M][N] (+=); swiglu: g [M][N/2]
  float* sumsq_out;         // resid: [M][N / kResGroup]
  __nv_bfloat16* xhl_out;   // resid: h * next_norm_w, swiglu: g, as hi, lo planes
  const __nv_bfloat16* next_norm_w;  // resid: [N]
  float* partials;          // [S][M][N] when S > 1
  unsigned* counters;       // [ceil(N / 128) + 1], zero on entry, left zero
  unsigned long long* amax_key;      // lmhead: [M]
  int32_t* argmax_out;               // lmhead: [M]
  unsigned* status;                  // time-out flag (may be null)
  // optional L2 prefetch of the next attention's cached K/V rows (as GemvParams); null: off
  const unsigned char* pf_kv;
  const int32_t* pf_positions;
  unsigned long long pf_plane_bytes, pf_head_bytes;
  int pf_B, pf_nkv, pf_row_bytes, pf_max_ctx;
};

// Fused q/k RMSNorm + RoPE + KV append + split-KV attention + LSE merge.
struct AttnParams {
  Timeline tl;
  // B rows = sequences x T tokens per sequence; row r is token r % T of sequence r / T
  // at position positions[r / T] + r % T (T <= 1: one row per sequence)
  int T;
  const float* qkv;             // [B][(nq + 2 nkv) d] projections
  const __nv_bfloat16* q_norm;  // [d]
  const __nv_bfloat16* k_norm;  // [d]
  const float2* rope;           // [B][d/2] (cos, sin) at this step's positions
  const int32_t* positions;     // [B / T] cached positions per sequence
  int kv_fmt;                   // DEC_KV_BF16 or DEC_KV_AFFINE8_G64
  __nv_bfloat16* kv;            // bf16 cache
  unsigned char* q8_codes;      // affine 8-bit cache: codes [L][2][B/T][nkv][max_ctx][d]
  unsigned char* q8_params;     //   and (scale, bias) bf16 pairs [L][2][B/T][nkv][max_ctx][d/64]
  int layer, B, nq, nkv, max_ctx;
  float eps;
  float* out;                   // [B][nq d]
  __nv_bfloat16* out_hl;        // optional: the output again as bf16 hi, lo planes [2][B][nq d]
  unsigned* status;
};

// On-device sampling of one token per row of logits (k_sample.cu).
constexpr int kSampleMaxK = 1024;  // candidates kept before top-p and the draw
struct SampleParams {
  const float* logits;  // [B][V]
  int V;
  float temperature;    // <= 0: greedy
  int top_k;            // 1..kSampleMaxK, else kSampleMaxK
  float top_p;          // (0, 1]; 1: no cut
  unsigned long long seed, offset;
  const unsigned long long* offset_dev;  // if not null, the offset is read here
  int32_t* tokens;      // [B]
};

struct EmbedParams {
  Timeline tl;
  const __nv_bfloat16* embed;   // [V][H]
  const int32_t* tokens;
  const int32_t* positions;
  const double* inv_freq;       // [d/2]
  float* h;                     // [B][H]
  float* sumsq;                 // [B][H / kResGroup]
  float2* rope;                 // [B][d/2]
  unsigned long long* amax_key; // [B]
  unsigned* status;
  const __nv_bfloat16* norm_w0;  // optional: first layer's input norm weight, for xhl_out
  __nv_bfloat16* xhl_out;        // optional: h * norm_w0 as bf16 hi, lo planes [2][B][H]
  int V, H, half_d, max_ctx;
  int T;                         // tokens per sequence: row b at position positions[b / T] + b % T
};

// ---------------------------------------------------------------- device helpers

__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Compiled in only when the library is built with DEC_TIMELINE=1: the stamps keep a
// predicate and a pointer live across the weight loop and cost the batch-1 GEMV 16
// registers, so the default build leaves them out.
__device__ __forceinline__ void tl_mark(const Timeline& tl, int slot) {
#if defined(DEC_TIMELINE) && DEC_TIMELINE
  if (tl.buf && threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (slot == 2)
      atomicMax(tl.buf + 3 * tl.idx + 2, t);
    else
      atomicMin(tl.buf + 3 * tl.idx + slot, t);
  }
#else
  (void)tl;
  (void)slot;
#endif
}
// Bulk prefetch of [src, src + bytes) into L2 (src and bytes multiples of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One CTA's share of the cached K/V rows (positions 0..P_b - 1 of every sequence b) that the
// next attention reads, prefetched into L2 by `nlanes` lanes: the 2 B nkv runs (plane,
// sequence, head) are dealt to the ncta CTAs round-robin, the CTAs of a run split it into equal
// 16-byte-aligned byte ranges, issued in pieces of at most 32 KB.
__device__ __forceinline__ void prefetch_kv_rows(const unsigned char* kv, const int32_t* positions,
                                                 unsigned long long plane_bytes, unsigned long long head_bytes,
                                                 int B, int nkv, int row_bytes, int max_ctx, int cta, int ncta,
                                                 int lane, int nlanes) {
  const int nruns = 2 * B * nkv;
  const int run = cta % nruns, slice = cta / nruns;
  const int nslices = (ncta - run + nruns - 1) / nruns;
  const int plane = run / (B * nkv), bh = run % (B * nkv), b = bh / nkv;
  int P = positions[b];
  P = P < 0 ? 0 : (P >= max_ctx ? max_ctx - 1 : P);
  const unsigned long long bytes = static_cast<unsigned long long>(P) * row_bytes;
  const unsigned long long per = ((bytes + nslices - 1) / nslices + 15) / 16 * 16;
  const unsigned long long off = per * slice;
  if (off >= bytes) return;
  const unsigned long long n = bytes - off < per ? bytes - off : per;
  const unsigned char* src = kv + plane * plane_bytes + bh * head_bytes + off;
  constexpr unsigned long long kPiece = 32768;
  const unsigned long long npieces = (n + kPiece - 1) / kPiece;
  for (unsigned long long i = lane; i < npieces; i += nlanes) {
    const unsigned long long o = i * kPiece;
    const unsigned long long m = n - o < kPiece ? n - o : kPiece;
    prefetch_l2_bulk(src + o, static_cast<uint32_t>(m));
  }
}

__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 16-byte streaming load that bypasses L1 (weights are read once per step).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Ordered-key encoding of a float so that unsigned comparison follows float order.
__device__ __forceinline__ uint32_t float_order_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  // larger value wins; among equal values the lower index wins (larger ~idx).  -0 and +0
  // compare equal as numbers, so -0 is keyed as +0 (adding +0 in round-to-nearest maps -0
  // to +0 and leaves every other value, NaN included, as it is).
  return (static_cast<unsigned long long>(float_order_key(__fadd_rn(v, 0.0f))) << 32) |
         static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(idx));
}
__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
}

// bf16x2 pack of two floats (round to nearest even), first argument in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------- tensor-core helpers (mma.sync)

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t smem_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t smem_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_addr));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes = 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace dec

// ---------------------------------------------------------------- host-side launchers
// (defined in the kernel translation units, called by the C-ABI layer)

namespace dec {

struct LaunchCtx {
  cudaStream_t stream;
  bool pdl;   // launch with programmatic stream serialization
};

cudaError_t launch_embed(const LaunchCtx& c, const EmbedParams& p, int B);
cudaError_t launch_gemv1(const LaunchCtx& c, const GemvParams& p, int wfmt, int in_mode, int epi);
cudaError_t launch_attention(const LaunchCtx& c, const AttnParams& p, int head_dim);
cudaError_t launch_kv_append(const LaunchCtx& c, const AttnParams& p, int head_dim);
// batched tensor-core projection
int gemm_tc_ny(int wfmt, int batch);            // 8-token n-tiles per hi/lo half, 0 if unsupported
int gemm_tc_block_tokens(int wfmt);             // most tokens one CTA takes (more: token blocks)
int gemm_tc_rows_per_block(int wfmt, int ny);   // weight rows one CTA covers
size_t gemm_tc_smem_bytes(int wfmt, int ny, int kc);
int gemm_tc_chunk(int ny);                      // inputs staged per chunk
cudaError_t launch_gemm_tc(const LaunchCtx& c, const GemmParams& p, int wfmt, int in_mode, int epi);
cudaError_t prepare_gemm_tc(const GemmParams& p, int wfmt, int in_mode, int epi);  // smem limit, before capture
// tcgen05 projections of many tokens (k_gemm_umma.cu)
int umma_tokens_per_tile();
int umma_k_step();
int umma_tile_n(int M, int N, int num_sms);  // weight rows per tile for an M x N projection
cudaError_t umma_tensor_map(void* map128, const void* ptr, int rows, int K, int box_rows);  // CUtensorMap (128 B)
cudaError_t launch_gemm_umma(const LaunchCtx& c, const void* map_x, const void* map_w, const UmmaParams& p,
                             int in_mode, int epi);
cudaError_t prepare_gemm_umma(int in_mode, int epi, int tile_n);
int q4tc_max_tokens();
int q4tc_splits(int N, int K, int num_sms);
cudaError_t q4tc_code_map(void* map128, const void* codes, int N, int K);  // CUtensorMap (128 B)
cudaError_t launch_gemm_q4tc(const LaunchCtx& c, const void* map_x, const void* map_codes, const Q4tcParams& p,
                             int in_mode, int epi);
cudaError_t prepare_gemm_q4tc(int in_mode, int epi);
// the bf16 form (k_gemm_btc.cu): the same parameters (sb unused), W bf16 [N][K] through a TMA
// map with 128-row boxes (umma_tensor_map)
cudaError_t launch_gemm_btc(const LaunchCtx& c, const void* map_x, const void* map_w, const Q4tcParams& p, int in_mode,
                            int epi);
cudaError_t prepare_gemm_btc(int in_mode, int epi);
int btc_max_segments(int N, int K, int ctas);  // partial-result slots of its stream-K schedule
int btc_box_rows(int M);                       // rows of its activation map's box for M tokens
// causal attention of prefill chunks (k_attn_prefill.cu): bf16 cache, head_dim 64 or 128,
// 1, 2 or 4 query heads per KV head; used from attn_prefill_min_tokens() tokens per sequence
int attn_prefill_min_tokens();
cudaError_t prepare_attn_prefill(int head_dim, int G);  // smem limit, before capture
cudaError_t launch_attn_prefill(const LaunchCtx& c, const AttnParams& p, int head_dim);
size_t attention_smem_bytes(int head_dim);
// set the dynamic smem limits and record the shapes' occupancy (before capture)
cudaError_t prepare_attention(int head_dim, int G, int kv_fmt);
// affine 8-bit cache kernels (k_attention_q8.cu)
cudaError_t prepare_attention_q8(int head_dim, int G, int (&max_clusters)[5]);
cudaError_t launch_attention_q8(const LaunchCtx& c, const AttnParams& p, int head_dim, int shape);
cudaError_t launch_kv_append_q8(const cudaLaunchConfig_t& cfg, const AttnParams& p, int head_dim);
cudaError_t launch_kv_quantize(cudaStream_t s, const float* src, int rows, int head_dim, unsigned char* codes,
                               __nv_bfloat16* params);

// Byte offset of the (scale, bias) pairs of an affine 8-bit cache: the codes, rounded up
// to 256 bytes.
inline size_t kv_q8_params_offset(const dec_config& c) {
  const size_t codes = static_cast<size_t>(c.n_layers) * 2 * c.batch * c.n_kv_heads * c.max_ctx * c.head_dim;
  return (codes + 255) / 256 * 256;
}

// The attention's view of a caller's cache in the config's format.
inline void attn_set_cache(AttnParams& ap, const dec_config& c, void* kv_cache) {
  ap.kv_fmt = c.kv_fmt;
  if (c.kv_fmt == DEC_KV_AFFINE8_G64) {
    ap.kv = nullptr;
    ap.q8_codes = static_cast<unsigned char*>(kv_cache);
    ap.q8_params = static_cast<unsigned char*>(kv_cache) + kv_q8_params_offset(c);
  } else {
    ap.kv = static_cast<__nv_bfloat16*>(kv_cache);
    ap.q8_codes = ap.q8_params = nullptr;
  }
}
// (cos, sin) of pos * theta^(-2i/d) for every sequence, angles and inverse
// frequencies in double on the device; out-of-range positions are clamped and flagged.
cudaError_t launch_rope_table(cudaStream_t s, const int32_t* positions, int batch, int head_dim, int max_ctx,
                              float theta, float2* rope, unsigned* status);

// create-time packing and test hooks
cudaError_t pack_rows_bf16(cudaStream_t s, __nv_bfloat16* dst, const __nv_bfloat16* src_a,
                           const __nv_bfloat16* src_b, int rows_out, int K, int interleave_block);
cudaError_t pack_rows_q4(cudaStream_t s, uint32_t* dst_w, uint32_t* dst_sb, const uint32_t* src_w_a,
                         const __nv_bfloat16* sc_a, const __nv_bfloat16* bi_a, const uint32_t* src_w_b,
                         const __nv_bfloat16* sc_b, const __nv_bfloat16* bi_b, int rows_out, int K,
                         int interleave_block);
cudaError_t debug_dequant(cudaStream_t s, float* out, const void* w, const uint32_t* sb, int wfmt,
                          int rows_out, int K, int row_offset, int interleave_block, int which_half);
// fragment-ordered packing for the batched path (rows padded with zeros to npad)
cudaError_t pack_frag_bf16(cudaStream_t s, uint32_t* dst, const __nv_bfloat16* src_a, const __nv_bfloat16* src_b,
                           int rows_out, int npad, int K, int interleave_block, int dst_row_offset, int dst_rows);
cudaError_t pack_frag_q4(cudaStream_t s, unsigned char* dst, const uint32_t* w_a, const __nv_bfloat16* sc_a,
                         const __nv_bfloat16* bi_a, const uint32_t* w_b, const __nv_bfloat16* sc_b,
                         const __nv_bfloat16* bi_b, int rows_out, int K, int interleave_block, int dst_row_offset,
                         int dst_rows);
cudaError_t debug_dequant_frag(cudaStream_t s, float* out, const void* w, int wfmt, int rows_out, int K,
                               int row_offset, int interleave_block, int which_half);
cudaError_t launch_hold(cudaStream_t s, unsigned long long ns);
cudaError_t launch_sample(cudaStream_t s, const SampleParams& p, int batch);
cudaError_t launch_force_timeout(cudaStream_t s, unsigned* status, int polls);
cudaError_t launch_advance(cudaStream_t s, const int32_t* argmax, int32_t* tokens, int32_t* positions,
                           int batch);

// Record the message returned by dec_last_error() on this thread.
void set_last_error(const char* fmt, ...);

// Argument checks of the stand-alone attention entry points (config limits, layer range,
// tokens_per_seq 0 or 1, kv_fmt); sets the last error and returns its status.
dec_status validate_attention_cfg(const dec_config* c, int layer);

}  // namespace dec

// Batch-1 fused GEMV kernels (CUDA cores): y = W x for one 8-row tile and one K split,
// with the RMSNorm of the input folded into the prologue and the consumer step
// (store / residual add / SwiGLU / lm_head argmax) folded into the epilogue.
//
// Butter architecture.md, "SINGLE-TOKEN DECODE": rms_norm -> gemv (q, k, v),
// gemv (o) -> add, rms_norm -> gemv (gate, up) -> silu_mul, gemv (down) -> add,
// rms_norm -> gemv (lm_head); the same page plans a fused rms_norm_qkv kernel
// that reads the activation once.  ANEForge "LLMs on the ANE", "lm_head on the
// ANE": the lm_head is tiled along the vocabulary; here each CTA is a vocab tile
// that reduces its own (max, index) and the last tile publishes the argmax.
//
// Weight streaming: every thread issues 16-byte L1-bypassing loads of 8 rows at
// once; the first chunk is requested before the grid-dependency wait, so it
// overlaps the previous kernel's tail (programmatic dependent launch).
//
// The input RMSNorm is linear in the product: y = rsqrt(mean(h^2) + eps) * W (h * w),
// so the loop runs on h * w and the scale is applied to the row sums at the end; the
// partial sums of squares are loaded right after the wait and reduced with the row
// sums, off the path to the first multiply.
//
// 4-bit decode: the codes of a word are split into even and odd bytes (two logic
// ops), each byte is moved into bits 16..19 of 128.0f by one byte permute (giving
// 128 + q exactly), and the products accumulate in pairs with the packed fp32 FMA
// (fma.rn.f32x2).  Per group: sum (s q + b) x = s sum (128 + q) x + (b - 128 s) sum x.
#include <type_traits>

#include "dec_internal.cuh"
#include "gemv_common.cuh"
#include "q4.cuh"

namespace dec {

namespace {

template <int WF>
struct ChunkTraits;
template <>
struct ChunkTraits<kWBf16> {
  static constexpr int kCols = 8;  // 16 bytes of bf16
};
template <>
struct ChunkTraits<kWQ4> {
  static constexpr int kCols = 16;  // 8 bytes of 4-bit codes (a quarter group): two words per row
};

template <int WF>
__device__ __forceinline__ const void* chunk_ptr(const GemvParams& p, int row, int col) {
  if constexpr (WF == kWBf16) {
    return static_cast<const __nv_bfloat16*>(p.w) + static_cast<size_t>(row) * p.K + col;
  } else {
    return static_cast<const uint32_t*>(p.w) + static_cast<size_t>(row) * (p.K / 8) + col / 8;
  }
}

using namespace gemv;

// This CTA's share of the next attention's cached K/V rows, prefetched into L2 by the
// lanes of one warp.  The 2 B n_kv runs (plane, sequence, head) of P_b rows each are
// dealt to the CTAs round-robin; the CTAs of a run split it into equal 16-byte-aligned
// byte ranges, issued in pieces of at most 32 KB.
__device__ __noinline__ void prefetch_kv_share(const GemvParams& p, int lane) {
  const int ncta = static_cast<int>(gridDim.x * gridDim.y);
  const int cta = static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x);
  const int nruns = 2 * p.pf_B * p.pf_nkv;
  const int run = cta % nruns, slice = cta / nruns;
  const int nslices = (ncta - run + nruns - 1) / nruns;
  const int plane = run / (p.pf_B * p.pf_nkv), bh = run % (p.pf_B * p.pf_nkv), b = bh / p.pf_nkv;
  int P = p.pf_positions[b];
  P = P < 0 ? 0 : (P >= p.pf_max_ctx ? p.pf_max_ctx - 1 : P);
  const unsigned long long bytes = static_cast<unsigned long long>(P) * p.pf_row_bytes;
  const unsigned long long per = ((bytes + nslices - 1) / nslices + 15) / 16 * 16;
  const unsigned long long off = per * slice;
  if (off >= bytes) return;
  const unsigned long long n = bytes - off < per ? bytes - off : per;
  const unsigned char* src = p.pf_kv + plane * p.pf_plane_bytes + bh * p.pf_head_bytes + off;
  constexpr unsigned long long kPiece = 32768;
  const unsigned long long npieces = (n + kPiece - 1) / kPiece;
  for (unsigned long long i = lane; i < npieces; i += 32) {
    const unsigned long long o = i * kPiece;
    const unsigned long long m = n - o < kPiece ? n - o : kPiece;
    prefetch_l2_bulk(src + o, static_cast<uint32_t>(m));
  }
}

}  // namespace

// Four CTAs of 256 threads per SM for bf16 (64 registers), three for the 4-bit decode.
template <int WF, int IN, int EPI>
__global__ void __launch_bounds__(256, (WF == kWBf16 ? 4 : 3)) k_gemv1(GemvParams p) {
  constexpr int R = kGemvRows;
  constexpr int CH = ChunkTraits<WF>::kCols;
  __shared__ float red[8][R + 1];  // per warp: R row sums, then the sum of squares
  __shared__ float ys[R];
  __shared__ float s_inv;
  __shared__ unsigned s_ticket;

  // Work units (row tile, K split), unit u = split * ntiles + tile; the CTAs take the
  // units round-robin and request the next unit's first chunk before reducing the
  // current one.
  const int ntiles = (p.N + R - 1) / R;
  const int nunits = ntiles * p.S;
  const int nchunk = p.KS / CH;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;

  tl_mark(p.tl, 0);
  using WReg = typename std::conditional<WF == kWBf16, uint4, uint2>::type;
  WReg wreg[R];
  uint32_t sbw[WF == kWQ4 ? R : 1];
  auto load_chunk = [&](int u, int cc) {
    const int tile = u % ntiles, row0 = tile * R, nrows = min(R, p.N - row0);
    const int col = (u / ntiles) * p.KS + cc * CH;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int row = row0 + min(r, nrows - 1);
      if constexpr (WF == kWBf16) {
        wreg[r] = ld_stream16(chunk_ptr<WF>(p, row, col));
      } else {
        wreg[r] = ld_stream8(chunk_ptr<WF>(p, row, col));
      }
      if constexpr (WF == kWQ4) sbw[r] = __ldg(p.sb + static_cast<size_t>(row) * (p.K / kGroup) + col / kGroup);
    }
  };
  // The first unit's first chunk (weights and 4-bit scale/bias words) does not depend
  // on upstream kernels: requested before the grid-dependency wait.
  int u = blockIdx.x;
  if (u < nunits && tid < nchunk) load_chunk(u, tid);
  if (p.pf_kv && warp == (nt >> 5) - 1) prefetch_kv_share(p, lane);
  // Residual rows of the first tile: last written two or more kernels upstream, which
  // completed before the previous kernel could pass its own wait and start this one.
  float h_pre = 0.f;
  if constexpr (EPI == kEpiResid) {
    if (tid < R && u < nunits) h_pre = __ldcg(p.out + (u % ntiles) * R + tid);
  }

  griddep_wait();
  tl_mark(p.tl, 1);

  // this thread's share of the input's partial sums of squares, reduced with the first
  // unit's row sums
  float ssq = 0.f;
  if constexpr (IN == kInNorm) {
    for (int i = tid; i < p.n_sumsq_in; i += nt) ssq += p.sumsq_in[i];
  }

  // 4-bit, one chunk per thread, no K split: a thread's input chunk (and its sum) is the
  // same in every unit and loaded once (bf16 reloads its 8 inputs: registers are tight).
  const bool x_fixed = WF == kWQ4 && p.S == 1 && nchunk <= nt;
  float xv[CH];
  float xsum = 0.f;
  __shared__ unsigned long long s_best;  // lm_head: this CTA's best (value, index) key
  if (tid == 0) s_best = 0ull;          // written and read by thread 0 only

  for (bool first = true; u < nunits; u += gridDim.x, first = false) {
    const int tile = u % ntiles, split = u / ntiles;
    const int row0 = tile * R;
    const int nrows = min(R, p.N - row0);
    const int kbeg = split * p.KS;
    const int un = u + gridDim.x;  // this CTA's next unit

    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;
    for (int c = tid; c < nchunk; c += nt) {
      const int col = kbeg + c * CH;
      if (first || !x_fixed) {
        load_x<IN, CH>(p, col, xv);
        if constexpr (WF == kWQ4) {
          xsum = 0.f;
#pragma unroll
          for (int i = 0; i < CH; ++i) xsum += xv[i];
        }
      }
      if constexpr (WF == kWBf16) {
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = dot_bf16x8(wreg[r], xv, acc[r]);
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float d0 = 0.f, d1 = 0.f;
          dot_q4_word(wreg[r].x, xv, d0, d1);
          dot_q4_word(wreg[r].y, xv + 8, d0, d1);
          const float s = sb_scale(sbw[r]), b = sb_bias(sbw[r]);
          acc[r] = fmaf(s, d0 + d1, acc[r]);
          acc[r] = fmaf(fmaf(-128.f, s, b), xsum, acc[r]);
        }
      }
      if (c + nt < nchunk) {
        load_chunk(u, c + nt);
      } else if (un < nunits) {
        load_chunk(un, tid);  // tid < nchunk here
      }
    }
    if (un >= nunits) griddep_launch_dependents();

    // block reduction of the R row sums (and, once, the sum of squares); fixed order:
    // lanes, then warps 0..n-1
    static_assert(R == 8, "warp_sum8 reduces 8 rows");
    {
      const float v = warp_sum8(acc, lane);
      if ((lane & 3) == 0) red[warp][lane >> 2] = v;
    }
    if (IN == kInNorm && first) {
      const float v = warp_sum(ssq);
      if (lane == 0) red[warp][R] = v;
    }
    __syncthreads();
    if (tid < R) {
      if (IN == kInNorm && first) {
        float q = 0.f;
        for (int w = 0; w < nt / 32; ++w) q += red[w][R];
        if (tid == 0) s_inv = rsqrtf(q / static_cast<float>(p.K) + p.eps);
      }
      float t = 0.f;
      for (int w = 0; w < nt / 32; ++w) t += red[w][tid];
      ys[tid] = t;
    }

    // split-K: the last CTA to finish a row tile adds the S partials in split order
    if (p.S > 1) {
      __syncthreads();
      if (tid < R && tid < nrows) {
        const float sc = IN == kInNorm ? s_inv : 1.f;
        p.partials[static_cast<size_t>(split) * p.N + row0 + tid] = ys[tid] * sc;
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) s_ticket = atomicAdd(&p.counters[tile], 1u);
      __syncthreads();
      if (s_ticket != static_cast<unsigned>(p.S - 1)) continue;
      __threadfence();
      if (tid < R && tid < nrows) {
        float t = 0.f;  // four splits requested at a time, added in split order
        for (int s0 = 0; s0 < p.S; s0 += 4) {
          float v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            v[j] = s0 + j < p.S ? __ldcg(p.partials + static_cast<size_t>(s0 + j) * p.N + row0 + tid) : 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) t += v[j];
        }
        ys[tid] = t;
      }
      if (tid == 0) p.counters[tile] = 0u;
    }
    __syncthreads();

    // epilogue: lane r of warp 0 owns row row0 + r; the other warps go on to the next unit
    if (warp != 0) continue;
    const bool mine = lane < R;
    float y = mine ? ys[lane] : 0.f;
    if (IN == kInNorm && p.S == 1) y *= s_inv;
    if constexpr (EPI == kEpiStore) {
      if (lane < nrows) p.out[row0 + lane] = y;
    } else if constexpr (EPI == kEpiResid) {
      float hn = 0.f;
      if (mine) {
        hn = (first ? h_pre : __ldcg(p.out + row0 + lane)) + y;
        p.out[row0 + lane] = hn;
      }
      float ss = hn * hn;  // the tile's 8 rows are one group of the norm's sums of squares
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      ss += __shfl_xor_sync(0xffffffffu, ss, 4);
      if (lane == 0) p.sumsq_out[tile] = ss;
    } else if constexpr (EPI == kEpiSwiglu) {
      // rows 0..3: gate of outputs 4 tile + i; rows 4..7: up of the same outputs
      const float up = __shfl_down_sync(0xffffffffu, y, R / 2);
      if (lane < R / 2) p.out[tile * (R / 2) + lane] = silu_f(y) * up;
    } else {  // lm_head tile: keep the CTA's best key, published once after the last unit
      if (lane < nrows && p.out) p.out[row0 + lane] = y;
      unsigned long long k = lane < nrows ? argmax_key(y, row0 + lane) : 0ull;
#pragma unroll
      for (int o = 1; o < R; o <<= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, k, o);
        k = other > k ? other : k;
      }
      if (lane == 0 && k > s_best) s_best = k;
    }
  }
  if constexpr (EPI == kEpiLmHead) {  // two-stage argmax: CTA keys, then the last CTA publishes
    if (tid == 0) {
      atomicMax(p.amax_key, s_best);
      __threadfence();
      const unsigned done = atomicAdd(&p.counters[ntiles], 1u);
      if (done == gridDim.x - 1) {
        __threadfence();
        const unsigned long long top = atomicOr(p.amax_key, 0ull);
        *p.argmax_out = argmax_key_index(top);
        p.counters[ntiles] = 0u;
      }
    }
  }
  if (lane == 0) tl_mark(p.tl, 2);
}

template <int WF, int IN, int EPI>
static cudaError_t launch_one(const LaunchCtx& c, const GemvParams& p) {
  constexpr int CH = ChunkTraits<WF>::kCols;
  const int nchunk = p.KS / CH;
  int nt = ((nchunk + 31) / 32) * 32;
  nt = nt < 32 ? 32 : (nt > 256 ? 256 : nt);
  // one wave of CTAs (every CTA resident at once), each looping over its units
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gemv1<WF, IN, EPI>, nt, 0)) != cudaSuccess)
    return e;
  const long long units = static_cast<long long>((p.N + kGemvRows - 1) / kGemvRows) * p.S;
  const long long cap = static_cast<long long>(per_sm > 0 ? per_sm : 1) * sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units < cap ? units : cap));
  cfg.blockDim = dim3(nt);
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemv1<WF, IN, EPI>, p);
}

cudaError_t launch_gemv1(const LaunchCtx& c, const GemvParams& p, int wfmt, int in_mode, int epi) {
#define DEC_GEMV_CASE(WF, IN, EPI) \
  if (wfmt == WF && in_mode == IN && epi == EPI) return launch_one<WF, IN, EPI>(c, p);
  DEC_GEMV_CASE(kWBf16, kInNorm, kEpiStore)
  DEC_GEMV_CASE(kWBf16, kInPlain, kEpiResid)
  DEC_GEMV_CASE(kWBf16, kInNorm, kEpiSwiglu)
  DEC_GEMV_CASE(kWBf16, kInNorm, kEpiLmHead)
  DEC_GEMV_CASE(kWQ4, kInNorm, kEpiStore)
  DEC_GEMV_CASE(kWQ4, kInPlain, kEpiResid)
  DEC_GEMV_CASE(kWQ4, kInNorm, kEpiSwiglu)
  DEC_GEMV_CASE(kWQ4, kInNorm, kEpiLmHead)
#undef DEC_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dec

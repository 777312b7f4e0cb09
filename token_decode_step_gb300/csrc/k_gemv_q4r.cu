// Batch-1 fused GEMV for affine 4-bit weights with the weight stream staged in shared memory:
// y = W x for 8-row tiles, the input RMSNorm folded into the prologue and the consumer step
// (store / residual add / SwiGLU / lm_head argmax) into the epilogue, as in k_gemv1.cu.
//
// Sources: oxinfer crate page, "MLX checkpoints" (the affine 4-bit format, eight codes per
// uint32 with a scale and bias per group of 64, and its per-group sum
// sum (s q + b) x = s sum q x + b sum x); Butter architecture.md, "SINGLE-TOKEN DECODE"
// (the projection sequence of one decode step and its fused kernels).
//
// The register-staged kernel keeps one unit of weights in flight per thread, so a CTA waits a
// whole DRAM latency for every unit and the decode instructions do not overlap the loads.  Here
// one producer thread per CTA streams whole units (8 rows x K/S inputs: the codes and the
// scale/bias words, one or sixteen bulk copies) into a ring of four shared-memory stages with
// cp.async.bulk, completing on an mbarrier per stage.  It needs no upstream result, so it fills
// the ring before the grid-dependency wait and keeps it full while the consumer warps decode:
// a consumer thread owns a 16-input chunk of the 8 rows (two words per row and the group's
// scale/bias word, all from shared memory), decodes with byte permutes into 128 + q and packed
// fp32 FMAs, and frees the stage with an mbarrier arrival.  The 8 row sums are reduced across
// the consumer warps (named barrier), split-K partials are added by the last CTA of a tile in
// split order.  Every wait on a barrier is bounded: on time-out the kernel flags the status
// word and stops waiting.
#include "gemv_common.cuh"
#include "umma_common.cuh"

namespace dec {

namespace {

using namespace gemv;
using umma::mbar_arrive;
using umma::mbar_expect_tx;
using umma::mbar_init;
using umma::mbar_wait;

constexpr int kR = kGemvRows;      // rows per unit
constexpr int kRStages = 4;        // shared-memory ring of units
constexpr int kRCols = 16;         // inputs per consumer chunk (two code words per row)
constexpr int kRMaxConsumers = 256;
constexpr int kRSmemMax = 200 * 1024;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void consumers_sync(int n) { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }

}  // namespace

template <int IN, int EPI>
__global__ void __launch_bounds__(kRMaxConsumers + 32) k_gemv_q4r(GemvParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red[kRMaxConsumers / 32][kR + 1];  // per warp: the 8 row sums, then the sum of squares
  __shared__ float ys[kR];
  __shared__ float s_inv;
  __shared__ unsigned s_ticket;
  __shared__ unsigned long long s_best;  // lm_head: this CTA's best (value, index) key

  const int KS = p.KS;
  const int code_bytes = kR * KS / 2, row_code = KS / 2, row_sb = KS / 16;
  const int stage_bytes = code_bytes + kR * row_sb;
  const uint32_t s_base = smem_u32(smem);
  const uint32_t full = s_base + kRStages * stage_bytes, empty = full + 8 * kRStages;
  const int ntiles = (p.N + kR - 1) / kR;
  const int nunits = ntiles * p.S;
  const int nchunk = KS / kRCols;
  const int ncons = static_cast<int>(blockDim.x) - 32;  // consumer threads; the last warp produces
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  tl_mark(p.tl, 0);
  if (tid == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, ncons);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_best = 0ull;
  }
  __syncthreads();

  bool ok = true;
  if (tid >= ncons) {
    // ---- producer: the weights do not depend on upstream kernels (no grid-dependency wait)
    if (lane == 0) {
      const int my_units = static_cast<int>(blockIdx.x) < nunits ? (nunits - 1 - blockIdx.x) / gridDim.x + 1 : 0;
      for (int i = 0; i < my_units; ++i) {
        const int u = blockIdx.x + i * gridDim.x, s = i % kRStages;
        if (i >= kRStages && !mbar_wait(empty + 8 * s, ((i / kRStages) - 1) & 1)) {
          ok = false;
          break;
        }
        const int tile = u % ntiles, split = u / ntiles;
        const int row0 = tile * kR, nrows = min(kR, p.N - row0);
        const uint32_t st = s_base + s * stage_bytes, bar = full + 8 * s;
        const unsigned char* wsrc =
            static_cast<const unsigned char*>(p.w) + static_cast<size_t>(row0) * (p.K / 2) + split * row_code;
        const unsigned char* ssrc =
            reinterpret_cast<const unsigned char*>(p.sb) + static_cast<size_t>(row0) * (p.K / 16) + split * row_sb;
        mbar_expect_tx(bar, static_cast<uint32_t>(nrows * (row_code + row_sb)));
        if (p.S == 1) {  // the tile's rows are contiguous: one copy of codes, one of scale/bias
          bulk_g2s(st, wsrc, static_cast<uint32_t>(nrows * row_code), bar);
          bulk_g2s(st + code_bytes, ssrc, static_cast<uint32_t>(nrows * row_sb), bar);
        } else {
          for (int r = 0; r < nrows; ++r) {
            bulk_g2s(st + r * row_code, wsrc + static_cast<size_t>(r) * (p.K / 2), static_cast<uint32_t>(row_code),
                     bar);
            bulk_g2s(st + code_bytes + r * row_sb, ssrc + static_cast<size_t>(r) * (p.K / 16),
                     static_cast<uint32_t>(row_sb), bar);
          }
        }
      }
    } else if (p.pf_kv) {  // the producer warp's other lanes: the next attention's K/V into L2
      prefetch_kv_rows(p.pf_kv, p.pf_positions, p.pf_plane_bytes, p.pf_head_bytes, p.pf_B, p.pf_nkv, p.pf_row_bytes,
                       p.pf_max_ctx, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), lane - 1, 31);
    }
    // No griddepcontrol.launch_dependents here: the first thread of a CTA to execute it
    // releases the dependent grid for that CTA, and a dependent reads data of the kernel
    // before this one (the residual) before its own wait, relying on this kernel having
    // passed its wait first.  The consumers release it after their wait.
  } else {
    // ---- consumers
    int u = blockIdx.x;
    // residual rows of the first tile: last written two or more kernels upstream, which
    // completed before the previous kernel could pass its own wait and start this one
    float h_pre = 0.f;
    if constexpr (EPI == kEpiResid) {
      if (tid < kR && u < nunits) h_pre = __ldcg(p.out + (u % ntiles) * kR + tid);
    }
    griddep_wait();
    tl_mark(p.tl, 1);
    float ssq = 0.f;  // this thread's share of the input's sums of squares
    if constexpr (IN == kInNorm) {
      for (int i = tid; i < p.n_sumsq_in; i += ncons) ssq += p.sumsq_in[i];
    }
    // one chunk per thread and no K split: the thread's input chunk is the same in every unit
    const bool x_fixed = p.S == 1 && nchunk <= ncons;
    float xv[kRCols];
    float xsum = 0.f;
    for (int it = 0; u < nunits; u += gridDim.x, ++it) {
      const bool first = it == 0;
      const int s = it % kRStages;
      const int tile = u % ntiles, split = u / ntiles;
      const int row0 = tile * kR, nrows = min(kR, p.N - row0);
      const int kbeg = split * KS;
      if (ok && !mbar_wait(full + 8 * s, (it / kRStages) & 1)) ok = false;
      const unsigned char* st = smem + s * stage_bytes;
      float acc[kR];
#pragma unroll
      for (int r = 0; r < kR; ++r) acc[r] = 0.f;
      for (int c = tid; c < nchunk; c += ncons) {
        if (first || !x_fixed) {
          load_x<IN, kRCols>(p, kbeg + c * kRCols, xv);
          xsum = 0.f;
#pragma unroll
          for (int i = 0; i < kRCols; ++i) xsum += xv[i];
        }
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          const int rr = r < nrows ? r : nrows - 1;
          const uint2 w = *reinterpret_cast<const uint2*>(st + rr * row_code + c * 8);
          const uint32_t sbw = *reinterpret_cast<const uint32_t*>(st + code_bytes + rr * row_sb + (c >> 2) * 4);
          float d0 = 0.f, d1 = 0.f;
          dot_q4_word(w.x, xv, d0, d1);
          dot_q4_word(w.y, xv + 8, d0, d1);
          const float sc = sb_scale(sbw), bi = sb_bias(sbw);
          acc[r] = fmaf(sc, d0 + d1, acc[r]);
          acc[r] = fmaf(fmaf(-128.f, sc, bi), xsum, acc[r]);
        }
      }
      mbar_arrive(empty + 8 * s);  // this thread's reads of the stage are done
      if (u + static_cast<int>(gridDim.x) >= nunits) griddep_launch_dependents();

      // reduction of the 8 row sums (and, once, the sum of squares); fixed order: lanes,
      // then warps 0..n-1
      {
        const float v = warp_sum8(acc, lane);
        if ((lane & 3) == 0) red[warp][lane >> 2] = v;
      }
      if (IN == kInNorm && first) {
        const float v = warp_sum(ssq);
        if (lane == 0) red[warp][kR] = v;
      }
      consumers_sync(ncons);
      if (tid < kR) {
        if (IN == kInNorm && first) {
          float q = 0.f;
          for (int w = 0; w < ncons / 32; ++w) q += red[w][kR];
          if (tid == 0) s_inv = rsqrtf(q / static_cast<float>(p.K) + p.eps);
        }
        float t = 0.f;
        for (int w = 0; w < ncons / 32; ++w) t += red[w][tid];
        ys[tid] = t;
      }
      if (p.S > 1) {  // the last CTA to finish a row tile adds the S partials in split order
        consumers_sync(ncons);
        if (tid < kR && tid < nrows) {
          const float sc = IN == kInNorm ? s_inv : 1.f;
          p.partials[static_cast<size_t>(split) * p.N + row0 + tid] = ys[tid] * sc;
        }
        __threadfence();
        consumers_sync(ncons);
        if (tid == 0) s_ticket = atomicAdd(&p.counters[tile], 1u);
        consumers_sync(ncons);
        if (s_ticket != static_cast<unsigned>(p.S - 1)) continue;
        __threadfence();
        if (tid < kR && tid < nrows) {
          float t = 0.f;
          for (int s2 = 0; s2 < p.S; ++s2) t += __ldcg(p.partials + static_cast<size_t>(s2) * p.N + row0 + tid);
          ys[tid] = t;
        }
        if (tid == 0) p.counters[tile] = 0u;
      }
      consumers_sync(ncons);

      // epilogue: lane r of warp 0 owns row row0 + r; the other warps go on to the next unit
      if (warp != 0) continue;
      const bool mine = lane < kR;
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
        const float up = __shfl_down_sync(0xffffffffu, y, kR / 2);
        if (lane < kR / 2) p.out[tile * (kR / 2) + lane] = silu_f(y) * up;
      } else {  // lm_head tile: keep the CTA's best key, published once after the last unit
        if (lane < nrows && p.out) p.out[row0 + lane] = y;
        unsigned long long k = lane < nrows ? argmax_key(y, row0 + lane) : 0ull;
#pragma unroll
        for (int o = 1; o < kR; o <<= 1) {
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
  }
  if (!ok && p.status) atomicOr(p.status, kStatusTimeout);
  if (lane == 0) tl_mark(p.tl, 2);
}

namespace {

size_t q4r_smem(int KS) { return static_cast<size_t>(kRStages) * (kR * KS / 2 + kR * KS / 16) + 16 * kRStages; }

template <int IN, int EPI>
cudaError_t q4r_launch(const LaunchCtx& c, const GemvParams& p, bool prepare) {
  if (prepare) return cudaFuncSetAttribute(k_gemv_q4r<IN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmemMax);
  const int nchunk = p.KS / kRCols;
  int cons = (nchunk + 31) / 32 * 32;
  cons = cons > kRMaxConsumers ? kRMaxConsumers : cons;
  const int nt = cons + 32;
  const size_t smem = q4r_smem(p.KS);
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gemv_q4r<IN, EPI>, nt, smem)) != cudaSuccess)
    return e;
  const long long units = static_cast<long long>((p.N + kR - 1) / kR) * p.S;
  const long long cap = static_cast<long long>(per_sm > 0 ? per_sm : 1) * sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units < cap ? units : cap));
  cfg.blockDim = dim3(nt);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemv_q4r<IN, EPI>, p);
}

cudaError_t q4r_dispatch(const LaunchCtx& c, const GemvParams& p, int in_mode, int epi, bool prepare) {
  if (in_mode == kInNorm && epi == kEpiStore) return q4r_launch<kInNorm, kEpiStore>(c, p, prepare);
  if (in_mode == kInPlain && epi == kEpiResid) return q4r_launch<kInPlain, kEpiResid>(c, p, prepare);
  if (in_mode == kInNorm && epi == kEpiSwiglu) return q4r_launch<kInNorm, kEpiSwiglu>(c, p, prepare);
  if (in_mode == kInNorm && epi == kEpiLmHead) return q4r_launch<kInNorm, kEpiLmHead>(c, p, prepare);
  return cudaErrorInvalidValue;
}

}  // namespace

// K splits for the staged kernel, 0 if the shape does not suit it: the bulk copies want each
// row's codes and scale/bias words of a split on 16-byte boundaries (K / S a multiple of 256)
// and a unit must fit a quarter of the staging memory.  Among those, the split count that
// minimises the bytes of the busiest SM (units dealt round-robin) plus a per-unit overhead,
// fewer splits on ties.
int gemv_q4r_splits(int N, int K, int num_sms) {
  if (K % 256 != 0 || num_sms <= 0) return 0;
  const long long tiles = (N + kR - 1) / kR;
  int best = 0;
  double best_cost = 0.0;
  for (int S = 1; S <= 8; ++S) {
    if (K % (256 * S) != 0) continue;
    const int KS = K / S;
    if (q4r_smem(KS) > static_cast<size_t>(kRSmemMax)) continue;
    const long long per_sm = (tiles * S + num_sms - 1) / num_sms;
    const double unit_bytes = kR * KS * 0.5625;
    const double cost = static_cast<double>(per_sm) * (unit_bytes + 2048.0);  // ~2 KB of DRAM time per unit
    if (best == 0 || cost < best_cost * 0.98) {
      best = S;
      best_cost = cost;
    }
  }
  return best;
}

cudaError_t prepare_gemv_q4r(int in_mode, int epi) {
  return q4r_dispatch(LaunchCtx{nullptr, false}, GemvParams{}, in_mode, epi, true);
}

cudaError_t launch_gemv_q4r(const LaunchCtx& c, const GemvParams& p, int in_mode, int epi) {
  return q4r_dispatch(c, p, in_mode, epi, false);
}

}  // namespace dec

// Batched decode projections with bf16 weights on the fifth-generation tensor cores:
// Y[t][n] = sum_k X[t][k] W[n][k] for up to 32 token rows (a batch of sequences, or the rows of
// a verify step).
//
// Sources: Butter architecture.md, "SINGLE-TOKEN DECODE" (the projection sequence, here over a
// batch of independent sequences).
//
// The 128 weight rows of a tile are the MMA's M (the accumulator's lanes) and the tokens' bf16
// hi and lo activation rows its N columns (16 + 16 rows up to 16 tokens, 32 + 32 beyond); both
// operands arrive by TMA as K-major tiles in the 128-byte swizzle, so the weights stream from
// HBM straight into the MMA's A operand.  The step is bound by that stream: one persistent CTA
// per SM keeps a ring of 8 or 10 weight tiles in flight, and two accumulators in tensor memory
// let the epilogue of one segment overlap the MMAs of the next.  Warp roles (192 threads): warp 0 issues the TMA copies, warp 1
// allocates the accumulators and issues the MMAs, warps 2..5 run the epilogue.
//
// Work is dealt stream-K: the tiles' 64-input stages, tile-major, are split into one contiguous
// range per CTA, so every SM streams the same number of weight bytes whatever the tile count
// (a whole-tile or K-split deal leaves the last wave part-empty: 384 units of the 8B gate/up on
// 152 SMs measured 49 us, 2.5 units a CTA).  A tile whose stages span several CTAs is computed
// in segments; each segment's partial result goes to a slot of the partial buffer and the last
// CTA to finish the tile adds the slots in K order (deterministic).  Every wait on a barrier is
// bounded: on time-out the kernel flags the status word and stops.
#include "tc_decode_epi.cuh"
#include "umma_common.cuh"

namespace dec {

namespace {

using namespace umma;

constexpr int kBM = 128;                  // weight rows per tile
constexpr int kBT = tcdec::kT;            // most token rows
constexpr int kBK = 64;                   // inputs per stage (one 128-byte row)
constexpr int kBW = kBM * kBK * 2;        // 16 KB: 128 weight rows of 128 bytes
constexpr int kBThreads = 192;
constexpr int kBSmemBudget = 200 * 1024;  // stage ring

// Activation tiles of MR rows (MR = 16 for up to 16 tokens, else 32): the hi rows, then the lo
// rows, are the MMA's N = 2 MR columns; the stage ring takes what the budget holds (10 stages
// at MR 16, 8 at MR 32), so fewer tokens keep more weight bytes in flight.
template <int MR>
struct BtcCfg {
  static constexpr int kX = 2 * MR * kBK * 2;
  static constexpr int kStage = kX + kBW;
  static constexpr int kStages = kBSmemBudget / kStage;
  static constexpr int kOffBar = kStages * kStage;
  static constexpr int kBars = 2 * kStages + 4;
  static constexpr int kOffTmem = kOffBar + 8 * kBars;
  static constexpr int kOffInv = kOffTmem + 16;
  static constexpr int kOffBest = kOffInv + 4 * kBT;
  static constexpr int kOffTicket = kOffBest + 8 * kBT;
  static constexpr int kSmem = 1024 + kOffTicket + 16;
  // tcgen05.mma kind::f16: fp32 accumulator, bf16 A and B, both K-major, N = 2 MR, M = 128
  static constexpr uint32_t kIdesc =
      (1u << 4) | (1u << 7) | (1u << 10) | ((static_cast<uint32_t>(2 * MR) >> 3) << 17) | ((128u >> 4) << 24);
  static_assert(kStage % 1024 == 0 && kX % 1024 == 0 && kOffBar % 8 == 0 && kOffBest % 8 == 0, "smem layout");
};

}  // namespace

template <int IN, int EPI, int MR>
__global__ void __launch_bounds__(kBThreads, 1)
    k_gemm_btc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, Q4tcParams p) {
  using CF = BtcCfg<MR>;
  constexpr int kBStages = CF::kStages, kBStage = CF::kStage, kBX = CF::kX;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms are 1024-byte aligned
  unsigned char* smem = smem_raw + (base - raw);
  const uint32_t st_full = base + CF::kOffBar, st_empty = st_full + 8 * kBStages;
  const uint32_t t_full = st_empty + 8 * kBStages, t_empty = t_full + 16;
  const uint32_t tmem_slot = base + CF::kOffTmem;
  float* s_inv = reinterpret_cast<float*>(smem + CF::kOffInv);
  unsigned long long* s_best = reinterpret_cast<unsigned long long*>(smem + CF::kOffBest);
  unsigned* s_ticket = reinterpret_cast<unsigned*>(smem + CF::kOffTicket);

  tl_mark(p.tl, 0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (p.N + kBM - 1) / kBM;
  const int kst = p.K / kBK;  // stages per tile
  const long long total = static_cast<long long>(n_tiles) * kst, grid = gridDim.x;
  const long long g_begin = tcdec::sk_begin(blockIdx.x, total, grid), g_end = tcdec::sk_begin(blockIdx.x + 1, total, grid);

  if (warp == 1) {  // two accumulators of 64 columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot), "r"(128)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(st_full + 8 * s, 1);
      mbar_init(st_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(t_full + 8 * b, 1);
      mbar_init(t_empty + 8 * b, 128);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (tid < kBT) s_best[tid] = 0ull;
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + CF::kOffTmem);

  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {  // TMA producer: stage i of this CTA is global stage g_begin + i
      const int nst = static_cast<int>(g_end - g_begin);
      // the weights do not depend on upstream kernels: the first stages' are requested before
      // the grid-dependency wait, their activations after it
      const int pre = nst < kBStages ? nst : kBStages;
      for (int i = 0; i < pre; ++i) {
        const long long g = g_begin + i;
        const uint32_t full = st_full + 8 * i, st = base + i * kBStage;
        mbar_expect_tx(full, kBStage);
        tma_load_2d(st + kBX, &tm_w, static_cast<int>(g % kst) * kBK, static_cast<int>(g / kst) * kBM, full);
      }
      griddep_wait();
      tl_mark(p.tl, 1);
      for (int i = 0; i < nst; ++i) {
        const long long g = g_begin + i;
        const int kb = static_cast<int>(g % kst), tile = static_cast<int>(g / kst);
        const int s = i % kBStages;
        const uint32_t full = st_full + 8 * s, st = base + s * kBStage;
        if (i >= pre) {
          if (!mbar_wait(st_empty + 8 * s, ((i / kBStages) - 1) & 1)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full, kBStage);
          tma_load_2d(st + kBX, &tm_w, kb * kBK, tile * kBM, full);
        }
        tma_load_2d(st, &tm_x, kb * kBK, 0, full);              // hi plane: tokens 0..MR-1
        tma_load_2d(st + kBX / 2, &tm_x, kb * kBK, p.M, full);  // lo plane
      }
    } else if (p.pf_kv) {  // the producer warp's other lanes: the next attention's K/V into L2
      prefetch_kv_rows(p.pf_kv, p.pf_positions, p.pf_plane_bytes, p.pf_head_bytes, p.pf_B, p.pf_nkv, p.pf_row_bytes,
                       p.pf_max_ctx, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), lane - 1, 31);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer: one accumulator per segment (a run of one tile's stages)
      int it = 0, local = 0;
      for (long long g = g_begin; g < g_end && ok; ++local) {
        const long long tile_end = (g / kst + 1) * kst, seg_end = tile_end < g_end ? tile_end : g_end;
        const int b = local & 1;
        if (local >= 2 && !mbar_wait(t_empty + 8 * b, ((local >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t acc = tmem + 64 * b;
        for (bool first = true; g < seg_end; ++g, ++it, first = false) {
          const int s = it % kBStages;
          if (!mbar_wait(st_full + 8 * s, (it / kBStages) & 1)) {
            ok = false;
            break;
          }
          fence_after();
          const uint32_t st = base + s * kBStage;
          const uint64_t dx = sw128_desc(st), dw = sw128_desc(st + kBX);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)  // 16 inputs = 32 bytes further along the swizzled rows
            mma_bf16(acc, dw + 2 * k, dx + 2 * k, CF::kIdesc, (!first || k != 0) ? 1u : 0u);
          commit(st_empty + 8 * s);
        }
        if (!ok) break;
        commit(t_full + 8 * b);
      }
    }
  } else {  // epilogue warps 2..5: accumulator lanes 32 q .. 32 q + 31, q = warp % 4
    const int et = tid - 64, q = warp & 3, r = 32 * q + lane;
    const uint32_t tq = static_cast<uint32_t>(32 * q) << 16;
    griddep_wait();  // the residual and the sums of squares are upstream outputs
    if constexpr (IN == kInNorm) {  // per-token 1/rms of the residual (the fused RMSNorm)
      if (warp == 2) {  // lane t sums token t's row of partial sums (a multiple of 8), independent loads
        float sacc = 0.f;
        if (lane < p.M) {
          const float4* row = reinterpret_cast<const float4*>(p.sumsq_in + static_cast<size_t>(lane) * p.n_sumsq_in);
          for (int k = 0; k < p.n_sumsq_in / 4; ++k) {
            const float4 v = __ldg(row + k);
            sacc += (v.x + v.y) + (v.z + v.w);
          }
        }
        s_inv[lane] = lane < p.M ? rsqrtf(sacc / static_cast<float>(p.K) + p.eps) : 0.f;
      }
    }
    tcdec::epi_sync();
    int local = 0;
    for (long long g = g_begin; g < g_end; ++local) {
      const int tile = static_cast<int>(g / kst), b = local & 1;
      const long long tile_end = static_cast<long long>(tile + 1) * kst;
      // the tile's segments: CTAs c_first .. c_last hold its stages, in K order
      const int c_first = tcdec::sk_cta_of(static_cast<long long>(tile) * kst, total, grid);
      const int c_last = tcdec::sk_cta_of(tile_end - 1, total, grid);
      g = tile_end < g_end ? tile_end : g_end;
      if (ok && !mbar_wait(t_full + 8 * b, (local >> 1) & 1)) ok = false;
      fence_after();
      float y[kBT], yl[kBT];
      tmem_ld32(tmem + 64 * b + tq, y);  // hi columns 0..MR-1, then lo columns
      if constexpr (MR == 32) tmem_ld32(tmem + 64 * b + 32 + tq, yl);
      fence_before();
      mbar_arrive(t_empty + 8 * b);
      if constexpr (MR == 32) {
#pragma unroll
        for (int t = 0; t < kBT; ++t) y[t] += yl[t];
      } else {
#pragma unroll
        for (int t = 0; t < MR; ++t) y[t] += y[MR + t];
#pragma unroll
        for (int t = MR; t < kBT; ++t) y[t] = 0.f;
      }
      const int n = tile * kBM + r;
      tcdec::unit_epilogue<IN, EPI, kBT, 128>(p, y, 0, n, tile, static_cast<int>(blockIdx.x) - c_first,
                                              c_last - c_first + 1, ok && n < p.N, et, lane, s_inv, s_best,
                                              s_ticket);
    }
    if constexpr (EPI == kEpiLmHead) {
      tcdec::epi_sync();
      if (et < p.M && s_best[et] != 0ull) atomicMax(p.amax_key + et, s_best[et]);
    }
  }
  griddep_launch_dependents();
  fence_before();
  __syncthreads();
  tl_mark(p.tl, 2);
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(128) : "memory");
  if (!ok && p.status) atomicOr(p.status, kStatusTimeout);
  if constexpr (EPI == kEpiLmHead) {  // the last CTA publishes every token's argmax
    __threadfence();
    if (tid == 0) *s_ticket = atomicAdd(&p.counters[n_tiles], 1u);
    __syncthreads();
    if (*s_ticket == gridDim.x - 1) {
      __threadfence();
      for (int bb = tid; bb < p.M; bb += kBThreads)
        p.argmax_out[bb] = argmax_key_index(atomicOr(p.amax_key + bb, 0ull));
      if (tid == 0) p.counters[n_tiles] = 0u;
    }
  }
}

namespace {

template <int IN, int EPI, int MR>
cudaError_t launch_btc_mr(const LaunchCtx& c, const CUtensorMap& mx, const CUtensorMap& mw, const Q4tcParams& p,
                          bool prepare) {
  constexpr int kSmem = BtcCfg<MR>::kSmem;
  if (prepare) return cudaFuncSetAttribute(k_gemm_btc<IN, EPI, MR>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  const long long stages = static_cast<long long>((p.N + kBM - 1) / kBM) * (p.K / kBK);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(stages < p.ctas ? stages : p.ctas));
  cfg.blockDim = dim3(kBThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemm_btc<IN, EPI, MR>, mx, mw, p);
}

template <int IN, int EPI>
cudaError_t launch_btc_t(const LaunchCtx& c, const CUtensorMap& mx, const CUtensorMap& mw, const Q4tcParams& p,
                         bool prepare) {
  if (prepare) {
    const cudaError_t e = launch_btc_mr<IN, EPI, 16>(c, mx, mw, p, true);
    return e != cudaSuccess ? e : launch_btc_mr<IN, EPI, 32>(c, mx, mw, p, true);
  }
  return p.M <= 16 ? launch_btc_mr<IN, EPI, 16>(c, mx, mw, p, false) : launch_btc_mr<IN, EPI, 32>(c, mx, mw, p, false);
}

cudaError_t dispatch_btc(const LaunchCtx& c, const CUtensorMap& mx, const CUtensorMap& mw, const Q4tcParams& p,
                         int in_mode, int epi, bool prepare) {
  if (in_mode == kInNorm && epi == kEpiStore) return launch_btc_t<kInNorm, kEpiStore>(c, mx, mw, p, prepare);
  if (in_mode == kInPlain && epi == kEpiStore) return launch_btc_t<kInPlain, kEpiStore>(c, mx, mw, p, prepare);
  if (in_mode == kInPlain && epi == kEpiResid) return launch_btc_t<kInPlain, kEpiResid>(c, mx, mw, p, prepare);
  if (in_mode == kInNorm && epi == kEpiSwiglu) return launch_btc_t<kInNorm, kEpiSwiglu>(c, mx, mw, p, prepare);
  if (in_mode == kInNorm && epi == kEpiLmHead) return launch_btc_t<kInNorm, kEpiLmHead>(c, mx, mw, p, prepare);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm_btc(const LaunchCtx& c, const void* map_x, const void* map_w, const Q4tcParams& p, int in_mode,
                            int epi) {
  return dispatch_btc(c, *static_cast<const CUtensorMap*>(map_x), *static_cast<const CUtensorMap*>(map_w), p, in_mode,
                      epi, false);
}

// Rows of the activation map's box (hi rows, then lo rows of a stage) for M tokens
int btc_box_rows(int M) { return M <= 16 ? 16 : 32; }

// Partial-result slots the stream-K schedule needs for an N x K projection on `ctas` CTAs: the
// most CTAs that share one tile (1: no tile is split)
int btc_max_segments(int N, int K, int ctas) {
  const long long n_tiles = (N + kBM - 1) / kBM, kst = K / kBK, total = n_tiles * kst;
  const long long grid = total < ctas ? total : ctas;
  int most = 1;
  for (long long t = 0; t < n_tiles; ++t) {
    const int segs = tcdec::sk_cta_of((t + 1) * kst - 1, total, grid) - tcdec::sk_cta_of(t * kst, total, grid) + 1;
    most = segs > most ? segs : most;
  }
  return most;
}

cudaError_t prepare_gemm_btc(int in_mode, int epi) {
  CUtensorMap dummy{};
  Q4tcParams p{};
  return dispatch_btc(LaunchCtx{nullptr, false}, dummy, dummy, p, in_mode, epi, true);
}

}  // namespace dec

// Projections of many tokens at once (prefill chunks) on the fifth-generation tensor cores:
// Y[t][n] = sum_k X[t][k] W[n][k] with tcgen05.mma, operands staged by the Tensor Memory
// Accelerator, the accumulator in tensor memory.
//
// Sources: Butter architecture.md, "SINGLE-TOKEN DECODE" (the projection sequence, here run
// over a chunk of prompt tokens); oxinfer crate page (prefill is compute-bound: a chunk of
// tokens reads the weights once).
//
// Tile: 128 tokens (the accumulator's 128 lanes) x 128 weight rows (128 fp32 columns), 64
// inputs per stage: one 128-byte row of bf16 per token and per weight row, so both operands
// are K-major tiles in the 128-byte swizzle that the TMA writes and the MMA reads.  The
// activations arrive as bf16 hi and lo planes (x = hi + lo, ~16 significant bits, the same
// planes the decode path's batched kernels read); both halves are multiplied into the same
// accumulator.  Four stages; one thread issues the TMA copies (full barriers complete on
// their bytes), one thread issues the MMAs (each stage's commit frees it for the copies),
// then all four warps read their 32 lanes of the accumulator for the epilogue.  Every wait
// on a barrier is bounded: on time-out the kernel flags the status word and leaves.
#include <cuda.h>

#include "umma_common.cuh"

namespace dec {

namespace {

constexpr int kUM = 128;                     // tokens per tile
constexpr int kUK = 64;                      // inputs per stage
constexpr int kUTile = 128 * kUK * 2;        // 16 KB: 128 rows of 128 bytes

// Per weight-tile width UN (128 or 256 rows = accumulator columns): the stage holds the x hi
// and lo tiles and UN weight rows; four stages of 48 KB, or three of 64 KB.
template <int UN>
struct UCfg {
  static constexpr int kStages = UN == 128 ? 4 : 3;
  static constexpr int kStage = 2 * kUTile + UN * kUK * 2;
  static constexpr int kSmem = 1024 + kStages * kStage + 256 + kUM * 4;
  // instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A and B, both
  // K-major, N = UN (N >> 3 at bit 17), M = 128 (M >> 4 at bit 24)
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((UN >> 3) << 17) | ((kUM >> 4) << 24);
};

using namespace umma;

__device__ __forceinline__ float silu_u(float x) { return x / (1.0f + expf(-x)); }

}  // namespace

// One 32-column chunk of a token's accumulator row (columns n0 .. n0 + 31, chunk c of weight
// tile nt): scale by the token's 1/rms, then the fused epilogue.
template <int IN, int EPI, int UN>
__device__ __forceinline__ void epi_chunk(const UmmaParams& p, float (&v)[32], int tok, int n0, int nt, int c,
                                          float r, unsigned long long& best) {
  constexpr int kUN = UN;
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] *= r;
  if constexpr (EPI == kEpiStore || EPI == kEpiLmHead) {
    if (p.out) {
      float* dst = p.out + static_cast<size_t>(tok) * p.N + n0;
      if (n0 + 32 <= p.N && (p.N & 3) == 0) {  // 16-byte aligned rows
#pragma unroll
        for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      } else {
        for (int i = 0; i < 32 && n0 + i < p.N; ++i) dst[i] = v[i];
      }
    }
    if constexpr (EPI == kEpiLmHead) {
      for (int i = 0; i < 32 && n0 + i < p.N; ++i) {
        const unsigned long long key = argmax_key(v[i], n0 + i);
        best = key > best ? key : best;
      }
    }
  } else if constexpr (EPI == kEpiResid) {
    // h += y; the next consumer's input h * next_norm as hi, lo planes; sums of squares per 8 rows
    float* hrow = p.out + static_cast<size_t>(tok) * p.N + n0;
    const size_t plane = static_cast<size_t>(p.M) * p.N;
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // groups of 8 rows (N is a multiple of 64)
      float ss = 0.f;
#pragma unroll
      for (int i = 8 * q; i < 8 * q + 8; ++i) {
        const float hn = hrow[i] + v[i];
        hrow[i] = hn;
        ss += hn * hn;
        const float x = hn * bf16_to_f(p.next_norm_w[n0 + i]);
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        const size_t o = static_cast<size_t>(tok) * p.N + n0 + i;
        p.xhl_out[o] = hi;
        p.xhl_out[plane + o] = __float2bfloat16_rn(x - __bfloat162float(hi));
      }
      p.sumsq_out[static_cast<size_t>(tok) * (p.N / kResGroup) + (n0 + 8 * q) / kResGroup] = ss;
    }
  } else {  // SwiGLU: columns 32 c .. 32 c + 15 are gate rows, the next 16 the matching up rows
    const int g0 = nt * (kUN / 2) + 16 * c;  // output index of the first pair
    const size_t plane = static_cast<size_t>(p.M) * (p.N / 2);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float gv = silu_u(v[i]) * v[16 + i];
      const size_t o = static_cast<size_t>(tok) * (p.N / 2) + g0 + i;
      p.out[o] = gv;
      const __nv_bfloat16 hi = __float2bfloat16_rn(gv);
      p.xhl_out[o] = hi;
      p.xhl_out[plane + o] = __float2bfloat16_rn(gv - __bfloat162float(hi));
    }
  }
}

// grid: (token tiles x weight-row tiles), token tiles fastest (the CTAs of one weight tile
// run together and share it through L2); 128 threads
template <int IN, int EPI, int UN>
__global__ void __launch_bounds__(128, 1)
    k_gemm_umma(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, UmmaParams p) {
  using CF = UCfg<UN>;
  constexpr int kUStages = CF::kStages, kUStage = CF::kStage, kUN = UN;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms are 1024-byte aligned
  unsigned char* smem = smem_raw + (base - raw);
  const uint32_t bar_full = base + kUStages * kUStage;
  const uint32_t bar_empty = bar_full + 8 * kUStages;
  const uint32_t bar_done = bar_empty + 8 * kUStages;
  const uint32_t tmem_slot = bar_done + 8;
  float* s_inv = reinterpret_cast<float*>(smem + kUStages * kUStage + 256);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = static_cast<int>(blockIdx.x) % p.m_tiles, nt = static_cast<int>(blockIdx.x) / p.m_tiles;

  if (warp == 0) {  // 128 accumulator columns (one CTA per SM: never contended)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot), "r"(kUN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 32) {
    for (int s = 0; s < kUStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + (tmem_slot - base));

  griddep_wait();  // the activations are the previous kernel's output
  if constexpr (IN == kInNorm) {  // per-token 1/rms of the residual (the fused RMSNorm)
    for (int j = 0; j < 32; ++j) {
      const int tok = mt * kUM + warp * 32 + j;
      float s = 0.f;
      if (tok < p.M)
        for (int i = lane; i < p.n_sumsq_in; i += 32) s += p.sumsq_in[static_cast<size_t>(tok) * p.n_sumsq_in + i];
      s = warp_sum(s);
      if (lane == 0) s_inv[warp * 32 + j] = rsqrtf(s / static_cast<float>(p.K) + p.eps);
    }
  }

  const int nk = p.K / kUK;
  bool ok = true;
  if (tid == 0) {  // TMA producer
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kUStages;
      if (kb >= kUStages && !mbar_wait(bar_empty + 8 * s, ((kb / kUStages) - 1) & 1)) {
        ok = false;
        break;
      }
      const uint32_t full = bar_full + 8 * s, st = base + s * kUStage;
      mbar_expect_tx(full, kUStage);
      tma_load_2d(st, &tm_x, kb * kUK, mt * kUM, full);
      tma_load_2d(st + kUTile, &tm_x, kb * kUK, p.M + mt * kUM, full);
      tma_load_2d(st + 2 * kUTile, &tm_w, kb * kUK, nt * kUN, full);
    }
  } else if (tid == 32) {  // MMA issuer
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kUStages;
      if (!mbar_wait(bar_full + 8 * s, (kb / kUStages) & 1)) {
        ok = false;
        break;
      }
      fence_after();
      const uint32_t st = base + s * kUStage;
      const uint64_t dxh = sw128_desc(st), dxl = sw128_desc(st + kUTile), dw = sw128_desc(st + 2 * kUTile);
#pragma unroll
      for (int k = 0; k < kUK / 16; ++k) {  // 16 inputs = 32 bytes further along the swizzled row
        mma_bf16(tmem, dxh + 2 * k, dw + 2 * k, CF::kIdesc, (kb | k) != 0 ? 1u : 0u);
        mma_bf16(tmem, dxl + 2 * k, dw + 2 * k, CF::kIdesc, 1u);
      }
      commit(bar_empty + 8 * s);  // the stage is free once these MMAs have read it
    }
    commit(bar_done);
  }
  __syncwarp();
  if (!mbar_wait(bar_done, 0)) ok = false;
  fence_after();
  __syncthreads();

  // ---- epilogue: this thread's token is lane 32 warp + lane of the tile
  const int tok = mt * kUM + warp * 32 + lane;
  const bool live = tok < p.M;
  const float r = (IN == kInNorm) ? s_inv[warp * 32 + lane] : 1.f;
  const uint32_t tlane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  unsigned long long best = 0ull;
#pragma unroll 1
  for (int c = 0; c < kUN / 32; ++c) {
    float v[32];
    tmem_ld32(tlane + 32 * c, v);  // (all lanes of the warp: the load is warp-collective)
    const int n0 = nt * kUN + 32 * c;
    // (N is a multiple of 32 for every epilogue but the lm_head's: a chunk is in or out)
    if (!live || !ok || n0 >= p.N) continue;
    epi_chunk<IN, EPI, UN>(p, v, tok, n0, nt, c, r, best);
  }
  if constexpr (EPI == kEpiLmHead) {
    if (live && ok) atomicMax(p.amax_key + tok, best);
  }
  griddep_launch_dependents();
  fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kUN) : "memory");
  if (!ok && tid == 0 && p.status) atomicOr(p.status, kStatusTimeout);
  if constexpr (EPI == kEpiLmHead) {  // the last CTA publishes every token's argmax
    __shared__ unsigned s_last;
    __threadfence();
    if (tid == 0) s_last = atomicAdd(&p.counters[0], 1u);
    __syncthreads();
    if (s_last == gridDim.x - 1) {
      __threadfence();
      for (int b = tid; b < p.M; b += 128) p.argmax_out[b] = argmax_key_index(atomicOr(p.amax_key + b, 0ull));
      if (tid == 0) p.counters[0] = 0u;
    }
  }
}

// Persistent form: one CTA per SM walks the tiles (token tiles fastest); warp 0 issues the
// TMA copies, warp 1 the MMAs, warps 2..5 run the epilogue.  Two accumulators in tensor
// memory: while the epilogue warps read tile i's, the MMAs of tile i + 1 fill the other
// (tmem_full: the MMA warp's commit after a tile; tmem_empty: 128 epilogue arrivals).
template <int IN, int EPI, int UN>
__global__ void __launch_bounds__(192, 1)
    k_gemm_umma_ps(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, UmmaParams p) {
  using CF = UCfg<UN>;
  constexpr int S = CF::kStages, kStage = CF::kStage;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  const uint32_t bar_full = base + S * kStage;
  const uint32_t bar_empty = bar_full + 8 * S;
  const uint32_t bar_tfull = bar_empty + 8 * S;   // [2]
  const uint32_t bar_tempty = bar_tfull + 16;     // [2]
  const uint32_t tmem_slot = bar_tempty + 16;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = p.m_tiles * ((p.N + UN - 1) / UN);
  const int nk = p.K / kUK;

  if (warp == 1) {  // two accumulators of UN columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot), "r"(2 * UN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 128);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + (tmem_slot - base));
  griddep_wait();

  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {  // TMA producer: the stage ring runs on across tiles
      int it = 0;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % S;
          if (it >= S && !mbar_wait(bar_empty + 8 * s, ((it / S) - 1) & 1)) {
            ok = false;
            break;
          }
          const uint32_t full = bar_full + 8 * s, st = base + s * kStage;
          mbar_expect_tx(full, kStage);
          tma_load_2d(st, &tm_x, kb * kUK, mt * kUM, full);
          tma_load_2d(st + kUTile, &tm_x, kb * kUK, p.M + mt * kUM, full);
          tma_load_2d(st + 2 * kUTile, &tm_w, kb * kUK, nt * UN, full);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      int it = 0, local = 0;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++local) {
        const int b = local & 1;
        if (local >= 2 && !mbar_wait(bar_tempty + 8 * b, ((local >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t acc = tmem + b * UN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % S;
          if (!mbar_wait(bar_full + 8 * s, (it / S) & 1)) {
            ok = false;
            break;
          }
          fence_after();
          const uint32_t st = base + s * kStage;
          const uint64_t dxh = sw128_desc(st), dxl = sw128_desc(st + kUTile), dw = sw128_desc(st + 2 * kUTile);
#pragma unroll
          for (int k = 0; k < kUK / 16; ++k) {
            mma_bf16(acc, dxh + 2 * k, dw + 2 * k, CF::kIdesc, (kb | k) != 0 ? 1u : 0u);
            mma_bf16(acc, dxl + 2 * k, dw + 2 * k, CF::kIdesc, 1u);
          }
          commit(bar_empty + 8 * s);
        }
        commit(bar_tfull + 8 * b);
      }
    }
  } else {  // epilogue warps 2..5: lanes 32 q .. 32 q + 31 of the accumulators, q = warp % 4
    const int q = warp & 3;
    const uint32_t tq = static_cast<uint32_t>(32 * q) << 16;
    unsigned long long best = 0ull;
    int local = 0, r_mt = -1;
    float r = 1.f;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++local) {
      const int mt = tile % p.m_tiles, nt = tile / p.m_tiles, b = local & 1;
      const int tok = mt * kUM + 32 * q + lane;
      const bool live = tok < p.M;
      if (IN == kInNorm && mt != r_mt) {  // the lane's token's 1/rms, once per token tile
        float sj = 0.f;
        if (live) {  // its row of partial sums (n_sumsq_in a multiple of 8), independent loads
          const float4* row = reinterpret_cast<const float4*>(p.sumsq_in + static_cast<size_t>(tok) * p.n_sumsq_in);
          for (int i = 0; i < p.n_sumsq_in / 4; ++i) {
            const float4 v = __ldg(row + i);
            sj += (v.x + v.y) + (v.z + v.w);
          }
        }
        r = rsqrtf(sj / static_cast<float>(p.K) + p.eps);
        r_mt = mt;
      }
      if (!mbar_wait(bar_tfull + 8 * b, (local >> 1) & 1)) ok = false;
      fence_after();
      if constexpr (EPI == kEpiLmHead) best = 0ull;
#pragma unroll 1
      for (int c = 0; c < UN / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + b * UN + tq + 32 * c, v);
        const int n0 = nt * UN + 32 * c;
        if (!live || !ok || n0 >= p.N) continue;
        epi_chunk<IN, EPI, UN>(p, v, tok, n0, nt, c, r, best);
      }
      fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_tempty + 8 * b) : "memory");
      if constexpr (EPI == kEpiLmHead) {
        if (live && ok) atomicMax(p.amax_key + tok, best);
      }
    }
  }
  griddep_launch_dependents();
  fence_before();
  __syncthreads();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * UN) : "memory");
  if (!ok && p.status) atomicOr(p.status, kStatusTimeout);
  if constexpr (EPI == kEpiLmHead) {  // the last CTA publishes every token's argmax
    __shared__ unsigned s_last;
    __threadfence();
    if (tid == 0) s_last = atomicAdd(&p.counters[0], 1u);
    __syncthreads();
    if (s_last == gridDim.x - 1) {
      __threadfence();
      for (int bb = tid; bb < p.M; bb += 192) p.argmax_out[bb] = argmax_key_index(atomicOr(p.amax_key + bb, 0ull));
      if (tid == 0) p.counters[0] = 0u;
    }
  }
}

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}

// bf16 [rows][K] row-major, boxes of 64 inputs x box_rows rows in the 128-byte swizzle;
// rows past the end read as zero
cudaError_t make_map(CUtensorMap* map, const void* ptr, int rows, int K, int box_rows) {
  EncodeTiled enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kUK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int IN, int EPI, int UN>
cudaError_t launch_umma_t(const LaunchCtx& c, const CUtensorMap& mx, const CUtensorMap& mw, const UmmaParams& p,
                          bool prepare) {
  auto kern = p.persistent ? k_gemm_umma_ps<IN, EPI, UN> : k_gemm_umma<IN, EPI, UN>;
  if (prepare) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_umma<IN, EPI, UN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         UCfg<UN>::kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_gemm_umma_ps<IN, EPI, UN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                UCfg<UN>::kSmem);
  }
  const int tiles = p.m_tiles * ((p.N + UN - 1) / UN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.persistent ? (tiles < p.persistent ? tiles : p.persistent) : tiles);
  cfg.blockDim = dim3(p.persistent ? 192 : 128);
  cfg.dynamicSmemBytes = UCfg<UN>::kSmem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mx, mw, p);
}

template <int UN>
cudaError_t dispatch_umma_n(const LaunchCtx& c, const CUtensorMap& mx, const CUtensorMap& mw, const UmmaParams& p,
                            int in_mode, int epi, bool prepare) {
  if (in_mode == kInNorm && epi == kEpiStore) return launch_umma_t<kInNorm, kEpiStore, UN>(c, mx, mw, p, prepare);
  if (in_mode == kInPlain && epi == kEpiStore) return launch_umma_t<kInPlain, kEpiStore, UN>(c, mx, mw, p, prepare);
  if (in_mode == kInPlain && epi == kEpiResid) return launch_umma_t<kInPlain, kEpiResid, UN>(c, mx, mw, p, prepare);
  if (in_mode == kInNorm && epi == kEpiSwiglu) return launch_umma_t<kInNorm, kEpiSwiglu, UN>(c, mx, mw, p, prepare);
  if (in_mode == kInNorm && epi == kEpiLmHead) return launch_umma_t<kInNorm, kEpiLmHead, UN>(c, mx, mw, p, prepare);
  return cudaErrorInvalidValue;
}

cudaError_t dispatch_umma(const LaunchCtx& c, const CUtensorMap& mx, const CUtensorMap& mw, const UmmaParams& p,
                          int in_mode, int epi, bool prepare) {
  if (p.tile_n == 256) return dispatch_umma_n<256>(c, mx, mw, p, in_mode, epi, prepare);
  if (p.tile_n == 128) return dispatch_umma_n<128>(c, mx, mw, p, in_mode, epi, prepare);
  return cudaErrorInvalidValue;
}

}  // namespace

int umma_tokens_per_tile() { return kUM; }
int umma_k_step() { return kUK; }

// 256-row weight tiles halve the activation re-reads per flop; 128-row tiles when 256 would
// leave SMs idle (small projections)
int umma_tile_n(int M, int N, int num_sms) {
  const long long m_tiles = (M + kUM - 1) / kUM;
  return m_tiles * ((N + 255) / 256) >= num_sms ? 256 : 128;
}

cudaError_t umma_tensor_map(void* map128, const void* ptr, int rows, int K, int box_rows) {
  static_assert(sizeof(CUtensorMap) == 128, "tensor map size");
  return make_map(static_cast<CUtensorMap*>(map128), ptr, rows, K, box_rows);
}

cudaError_t launch_gemm_umma(const LaunchCtx& c, const void* map_x, const void* map_w, const UmmaParams& p,
                             int in_mode, int epi) {
  return dispatch_umma(c, *static_cast<const CUtensorMap*>(map_x), *static_cast<const CUtensorMap*>(map_w), p,
                       in_mode, epi, false);
}

cudaError_t prepare_gemm_umma(int in_mode, int epi, int tile_n) {
  CUtensorMap dummy{};
  UmmaParams p{};
  p.tile_n = tile_n;
  return dispatch_umma(LaunchCtx{nullptr, false}, dummy, dummy, p, in_mode, epi, true);
}

}  // namespace dec

// Batched decode projections with affine 4-bit weights on the fifth-generation tensor cores:
// Y[t][n] = sum_k X[t][k] W[n][k] for up to 32 token rows, W = scale * q + bias per group of
// 64 inputs (q in 0..15, eight per uint32, one bf16 scale and bias per group).
//
// Sources: oxinfer crate page, "MLX checkpoints" (the affine 4-bit format and its per-group
// sum: sum_k (s q_k + b) x_k = s sum_k q_k x_k + b sum_k x_k); Butter architecture.md,
// "SINGLE-TOKEN DECODE" (the projection sequence, here over a batch of independent sequences).
//
// Per group of 64 inputs the tensor cores compute D[n][t] = sum_k (128 + q[n][k]) x[t][k] with
// the codes as exact bf16 integers: a tile's 120 weight rows and 8 rows of ones are the MMA's
// M = 128 (the accumulator's lanes) and its A operand, which the expanding threads write straight
// into tensor memory (row n in lane n, two codes per 32-bit column); the activations' 32 bf16 hi
// rows and 32 lo rows are its N = 64 columns (B, K-major in the 128-byte swizzle, read from
// shared memory).  The rows of ones give each token's sum of the group's inputs in the same
// instruction.  The epilogue warps read every group's accumulator from a ring in tensor memory
// and add s D (hi and lo columns) and (b - 128 s) sum_k x[t][k] in float32, in a fixed order (per
// stage the s D terms of its groups, then their sum-of-x terms), so the scale and bias cost one
// multiply-add each per (row, token, group) instead of a dequantization per weight.
//
// Warp roles (one persistent CTA per SM, 576 threads), handing over stages of two groups
// (halving the barrier round trips per byte): warp 0 issues the TMA copies of the codes (120
// rows x 64 bytes a stage) and of the activation tiles (32 hi rows, 32 lo rows per group);
// warp 1 allocates tensor memory and issues the MMAs; warps 2..9 expand the codes into bf16 (a
// byte permute builds 128 + q for two codes) and store them to the A ring in tensor memory;
// warps 10..17 scale, accumulate and run the fused epilogue, two warps per 32-lane quarter of
// the accumulator, 16 tokens each.
// A unit is a (120-row tile, K split) pair; with S > 1 splits the last CTA to finish a tile
// adds the S partial results in split order (deterministic).  Every wait on a barrier is
// bounded: on time-out the kernel flags the status word and stops.
#include "q4.cuh"
#include "tc_decode_epi.cuh"
#include "umma_common.cuh"

namespace dec {

namespace {

using namespace umma;

constexpr int kQM = 128;                   // MMA rows: accumulator lanes
constexpr int kQRows = 120;                // weight rows per tile; lanes 120..127 are rows of ones
constexpr int kQT = 32;                    // token rows (accumulator columns)
constexpr int kQK = 64;                    // inputs per group of the format
constexpr int kQSG = 2;                    // groups per stage: every hand-off covers two groups
constexpr int kQN = 2 * kQT;               // MMA N: the hi rows, then the lo rows, of the tokens
constexpr int kQStages = 6;                // TMA ring: codes + activations, of kQSG groups each
constexpr int kQAStages = 2;               // expanded-code ring in tensor memory (stages)
constexpr int kQG = 3;                     // accumulator ring (stages of kQSG x 64 columns)
constexpr int kQACols = kQK / 2;           // 32 columns: a group of 64 bf16 codes per lane
constexpr int kQAOff = kQN * kQSG * kQG;   // first column of the code ring
constexpr int kQTmemCols = 512;            // kQAOff + kQAStages * kQSG * kQACols
constexpr int kQCodeRow = kQSG * kQK / 2;  // 64 bytes of codes per row and stage
constexpr int kQCode = kQM * kQCodeRow;    // 8 KB slot: kQRows rows x 64 bytes of codes
constexpr int kQXg = 2 * kQT * kQK * 2;    // 8 KB per group: 32 hi rows, then 32 lo rows, of 128 bytes
constexpr int kQX = kQSG * kQXg;
constexpr int kQStage = kQX + kQCode;      // activations first (1024-byte aligned atoms)
constexpr int kQCodeTx = kQRows * kQCodeRow;  // bytes of a stage's code box
constexpr int kQDefer = 1;                 // stage of the next unit after which a split exchange runs
constexpr int kQDeq = 256;                 // expansion threads
constexpr int kQEpi = 256;                 // epilogue threads
constexpr int kQThreads = 64 + kQDeq + kQEpi;
constexpr int kQOffS = 0;
constexpr int kQOffBar = kQOffS + kQStages * kQStage;
constexpr int kQBars = 2 * kQStages + 2 * kQAStages + 2 * kQG;
constexpr int kQOffTmem = kQOffBar + 8 * kQBars;
constexpr int kQOffSx = kQOffTmem + 16;  // float [2][kQSG][kQT]: sums of x, by stage parity
constexpr int kQOffInv = kQOffSx + 4 * 2 * kQSG * kQT;
constexpr int kQOffBest = kQOffInv + 4 * kQT;
constexpr int kQOffTicket = kQOffBest + 8 * kQT;
constexpr int kQSmem = 1024 + kQOffTicket + 16;
// tcgen05.mma kind::f16: fp32 accumulator, bf16 A and B, both K-major, N = 64, M = 128
constexpr uint32_t kQIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((static_cast<uint32_t>(kQN) >> 3) << 17) |
                             ((128u >> 4) << 24);
static_assert(kQAOff + kQAStages * kQSG * kQACols <= kQTmemCols, "tensor memory layout");
static_assert(kQOffS % 1024 == 0 && kQStage % 1024 == 0 && kQOffBar % 8 == 0 && kQOffBest % 8 == 0, "smem layout");

using tcdec::epi_sync;

// Codes of one word (element 8 j + k in bits 4k..4k+3) -> the 16 bytes of bf16 (128 + q) for
// elements 8 j .. 8 j + 7 in order.  The permutes interleave even and odd codes and set 0x43
// as each high byte: bf16 0x43qq is 128 + q exactly.  (The products then accumulate in float32
// at about 17 times the magnitude of centred codes: rounding stays near 1e-7 of the bound.)
__device__ __forceinline__ uint4 expand_word(uint32_t w) {
  const uint32_t ev = w & 0x0f0f0f0fu, od = (w >> 4) & 0x0f0f0f0fu;  // codes 0,2,4,6 / 1,3,5,7
  const uint32_t t0 = __byte_perm(ev, od, 0x5140), t1 = __byte_perm(ev, od, 0x7362);  // c0..c3 / c4..c7
  constexpr uint32_t k43 = 0x43434343u;
  return make_uint4(__byte_perm(t0, k43, 0x4140), __byte_perm(t0, k43, 0x4342), __byte_perm(t1, k43, 0x4140),
                    __byte_perm(t1, k43, 0x4342));
}

// (y0, y1) += (a0, a1) * (b0, b1), one packed float32 FMA
__device__ __forceinline__ void fma2(float& y0, float& y1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b, y;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %5};\n\t"
      "mov.b64 y, {%0, %1};\n\t"
      "fma.rn.f32x2 y, a, b, y;\n\t"
      "mov.b64 {%0, %1}, y;\n\t}"
      : "+f"(y0), "+f"(y1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

}  // namespace

template <int IN, int EPI>
__global__ void __launch_bounds__(kQThreads, 1)
    k_gemm_q4tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_c, Q4tcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms are 1024-byte aligned
  unsigned char* smem = smem_raw + (base - raw);
  const uint32_t sS = base + kQOffS;
  const uint32_t st_full = base + kQOffBar, st_empty = st_full + 8 * kQStages;
  const uint32_t a_full = st_empty + 8 * kQStages, a_empty = a_full + 8 * kQAStages;
  const uint32_t g_full = a_empty + 8 * kQAStages, g_empty = g_full + 8 * kQG;
  const uint32_t tmem_slot = base + kQOffTmem;
  float* s_x = reinterpret_cast<float*>(smem + kQOffSx);
  float* s_inv = reinterpret_cast<float*>(smem + kQOffInv);
  unsigned long long* s_best = reinterpret_cast<unsigned long long*>(smem + kQOffBest);
  unsigned* s_ticket = reinterpret_cast<unsigned*>(smem + kQOffTicket);

  tl_mark(p.tl, 0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (p.N + kQRows - 1) / kQRows;
  const int units = n_tiles * p.S;
  const int gps = p.K / kQK / p.S;  // groups per split
  const int spu = (gps + kQSG - 1) / kQSG;  // stages per unit; with gps odd the last holds one group

  if (warp == 1) {  // the accumulator ring (kQG x kQSG x 64 columns), then the code ring
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot), "r"(kQTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(st_full + 8 * s, 1);
      mbar_init(st_empty + 8 * s, kQDeq + 1);  // the expanders' reads, then the MMAs' commit
    }
    for (int s = 0; s < kQAStages; ++s) {
      mbar_init(a_full + 8 * s, kQDeq);
      mbar_init(a_empty + 8 * s, 1);
    }
    for (int b = 0; b < kQG; ++b) {
      mbar_init(g_full + 8 * b, 1);     // the MMAs' commit
      mbar_init(g_empty + 8 * b, kQEpi);  // the epilogue's accumulator reads
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (tid < kQT) s_best[tid] = 0ull;
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kQOffTmem);

  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {  // TMA producer; stage i of this CTA holds groups 2 (i % spu) .. of its unit i / spu
      const int my_units = static_cast<int>(blockIdx.x) < units ? (units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
      const int total = my_units * spu;
      auto stage_of = [&](int i, int& tile, int& g0, int& ng) {
        const int u = blockIdx.x + (i / spu) * gridDim.x, js = i % spu;
        tile = u % n_tiles;
        g0 = (u / n_tiles) * gps + kQSG * js;
        ng = gps - kQSG * js < kQSG ? gps - kQSG * js : kQSG;
      };
      // the codes do not depend on upstream kernels: the first stages' are requested before
      // the grid-dependency wait, their activations after it (a code box always spans kQSG
      // groups; past the end of a split it reads codes that are not used, past K zeros)
      const int pre = total < kQStages ? total : kQStages;
      for (int i = 0; i < pre; ++i) {
        int tile, g0, ng;
        stage_of(i, tile, g0, ng);
        const uint32_t full = st_full + 8 * i, st = sS + i * kQStage;
        mbar_expect_tx(full, kQCodeTx + ng * kQXg);
        tma_load_2d(st + kQX, &tm_c, g0 * (kQK / 2), tile * kQRows, full);
      }
      griddep_wait();
      tl_mark(p.tl, 1);
      for (int i = 0; i < total; ++i) {
        int tile, g0, ng;
        stage_of(i, tile, g0, ng);
        const int s = i % kQStages;
        const uint32_t full = st_full + 8 * s, st = sS + s * kQStage;
        if (i >= pre) {
          if (!mbar_wait(st_empty + 8 * s, ((i / kQStages) - 1) & 1)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full, kQCodeTx + ng * kQXg);
          tma_load_2d(st + kQX, &tm_c, g0 * (kQK / 2), tile * kQRows, full);
        }
        for (int gg = 0; gg < ng; ++gg) {
          tma_load_2d(st + gg * kQXg, &tm_x, (g0 + gg) * kQK, 0, full);                // hi plane: tokens 0..31
          tma_load_2d(st + gg * kQXg + kQXg / 2, &tm_x, (g0 + gg) * kQK, p.M, full);  // lo plane
        }
      }
    } else if (p.pf_kv) {  // the producer warp's other lanes: the next attention's K/V into L2
      prefetch_kv_rows(p.pf_kv, p.pf_positions, p.pf_plane_bytes, p.pf_head_bytes, p.pf_B, p.pf_nkv, p.pf_row_bytes,
                       p.pf_max_ctx, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), lane - 1, 31);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer: one accumulator per group, kQSG of them per stage
      int it = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        for (int js = 0; js < spu; ++js, ++it) {
          const int s = it % kQStages, a = it % kQAStages, gb = it % kQG;
          const int ng = gps - kQSG * js < kQSG ? gps - kQSG * js : kQSG;
          if (!mbar_wait(a_full + 8 * a, (it / kQAStages) & 1) || !mbar_wait(st_full + 8 * s, (it / kQStages) & 1) ||
              (it >= kQG && !mbar_wait(g_empty + 8 * gb, ((it / kQG) - 1) & 1))) {
            ok = false;
            break;
          }
          fence_after();
          // D[n][0..31] = sum (128 + q) x_hi, D[n][32..63] = sum (128 + q) x_lo; A from tensor memory
          for (int gg = 0; gg < ng; ++gg) {
            const uint64_t dx = sw128_desc(sS + s * kQStage + gg * kQXg);
            const uint32_t ta = tmem + kQAOff + kQACols * (kQSG * a + gg);
            const uint32_t td = tmem + kQN * (kQSG * gb + gg);
#pragma unroll
            for (int k = 0; k < kQK / 16; ++k)  // 16 inputs: 8 columns of A, 32 bytes along the swizzled B rows
              mma_bf16_ta(td, ta + 8 * k, dx + 2 * k, kQIdesc, k != 0 ? 1u : 0u);
          }
          commit(a_empty + 8 * a);
          commit(st_empty + 8 * s);
          commit(g_full + 8 * gb);
        }
      }
    }
  } else if (warp < 10) {
    // expanders: weight row r = 32 (warp % 4) + lane of the tile (the tensor-memory lanes this
    // warp may write), inputs 32 h .. 32 h + 31 of each group.  Lanes 120..127 store ones instead:
    // the accumulator's lanes there then hold each token's sum of the group's inputs.
    const int r = 32 * (warp & 3) + lane, h = (warp - 2) >> 2;
    const bool ones = r >= kQRows;
    const uint32_t ta_row = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + kQAOff + 16 * h;
    int it = 0;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      for (int js = 0; js < spu; ++js, ++it) {
        const int s = it % kQStages, a = it % kQAStages;
        const int ng = gps - kQSG * js < kQSG ? gps - kQSG * js : kQSG;
        // waits are made warp-uniform: the tensor-memory stores below are whole-warp instructions
        if (!__all_sync(0xffffffffu, mbar_wait(st_full + 8 * s, (it / kQStages) & 1))) {
          ok = false;
          break;
        }
        uint4 cw[kQSG];
#pragma unroll
        for (int gg = 0; gg < kQSG; ++gg) {
          cw[gg] = make_uint4(0u, 0u, 0u, 0u);
          if (!ones && gg < ng)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(cw[gg].x), "=r"(cw[gg].y), "=r"(cw[gg].z), "=r"(cw[gg].w)
                         : "r"(sS + s * kQStage + kQX + r * kQCodeRow + gg * (kQK / 2) + h * 16));
        }
        mbar_arrive(st_empty + 8 * s);
        if (it >= kQAStages && !__all_sync(0xffffffffu, mbar_wait(a_empty + 8 * a, ((it / kQAStages) - 1) & 1))) {
          ok = false;
          break;
        }
        fence_after();
#pragma unroll
        for (int gg = 0; gg < kQSG; ++gg) {
          if (gg >= ng) break;  // ng is the same for the whole warp
          uint32_t v[16];  // inputs 32 h + 2 j, 32 h + 2 j + 1 in column j (low half first)
          const uint32_t words[4] = {cw[gg].x, cw[gg].y, cw[gg].z, cw[gg].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 e = expand_word(words[i]);
            v[4 * i] = e.x;
            v[4 * i + 1] = e.y;
            v[4 * i + 2] = e.z;
            v[4 * i + 3] = e.w;
          }
          if (ones) {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0x3F803F80u;  // bf16 1.0 in both halves
          }
          tmem_st16(ta_row + kQACols * (kQSG * a + gg), v);
        }
        fence_before();
        mbar_arrive(a_full + 8 * a);
      }
    }
  } else {  // epilogue warps 10..17: accumulator lanes 32 q .. 32 q + 31 (q = warp % 4), columns 16 c .. 16 c + 15
    const int et = tid - 64 - kQDeq, q = warp & 3, c = (warp - 10) >> 2, r = 32 * q + lane;
    const uint32_t tq = static_cast<uint32_t>(32 * q) << 16;
    constexpr int kTPT = kQT / 2;  // token columns per thread
    griddep_wait();  // the residual and the sums of squares are upstream outputs
    if constexpr (IN == kInNorm) {  // per-token 1/rms of the residual (the fused RMSNorm)
      if (warp == 10) {  // lane t sums token t's row of partial sums (a multiple of 8), independent loads
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
    epi_sync<kQEpi>();
    // With K splits a unit's partial results are written at its end and the exchange (fence,
    // ticket, and in the tile's last CTA the sum of the slots and the fused epilogue) waits
    // until the next unit's first groups are under way: done at once, its round trips stalled
    // the epilogue while the rings filled and the MMAs and expansion stopped behind it.
    int pend_tile = -1, pend_n = 0;
    bool pend_live = false;
    auto finish_pending = [&]() {
      float yp[kTPT];
      if (tcdec::split_finish<kTPT, kQEpi>(p, yp, kTPT * c, pend_n, pend_tile, p.S, pend_live, et, s_ticket))
        tcdec::fused_epilogue<IN, EPI, kTPT>(p, yp, kTPT * c, pend_n, pend_live, lane, s_inv, s_best);
      pend_tile = -1;
    };
    int it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int tile = u % n_tiles, split = u / n_tiles;
      const int n = tile * kQRows + r;
      const bool row_ok = r < kQRows && n < p.N;
      const uint32_t* sbrow = p.sb + static_cast<size_t>(row_ok ? n : 0) * (p.K / kGroup) + split * gps;
      float y[kTPT];
#pragma unroll
      for (int t = 0; t < kTPT; ++t) y[t] = 0.f;
      uint32_t sbw[kQSG], sbn[kQSG];  // this stage's scale/bias words; the next stage's, in flight
#pragma unroll
      for (int gg = 0; gg < kQSG; ++gg) sbw[gg] = gg < gps ? __ldg(sbrow + gg) : 0u;
      for (int js = 0; js < spu; ++js, ++it) {
        const int gb = it % kQG, j0 = kQSG * js;
        const int ng = gps - j0 < kQSG ? gps - j0 : kQSG;
#pragma unroll
        for (int gg = 0; gg < kQSG; ++gg) sbn[gg] = j0 + kQSG + gg < gps ? __ldg(sbrow + j0 + kQSG + gg) : 0u;
        if (ok && !mbar_wait(g_full + 8 * gb, (it / kQG) & 1)) ok = false;
        fence_after();
        // w = s q + b = s (128 + q) + (b - 128 s): y += s D_hi + s D_lo, per group, now; the
        // (b - 128 s) sum x terms after the barrier that publishes the sums.  The first ones
        // lane holds each group's sums of x and publishes them for the other lanes (two buffers
        // by stage parity; the barrier of stage it - 1 orders these writes after every read of
        // stage it - 2).
        float* sx = s_x + (it & 1) * (kQSG * kQT) + kTPT * c;
#pragma unroll
        for (int gg = 0; gg < kQSG; ++gg) {
          if (gg >= ng) break;  // ng is the same for every epilogue thread
          float d[kTPT], dl[kTPT];
          const uint32_t td = tmem + kQN * (kQSG * gb + gg) + kTPT * c + tq;
          tmem_ld16(td, d);         // hi columns of tokens 16 c .. 16 c + 15
          tmem_ld16(td + kQT, dl);  // their lo columns
          if (r == kQRows) {
#pragma unroll
            for (int t4 = 0; t4 < kTPT / 4; ++t4)
              reinterpret_cast<float4*>(sx + gg * kQT)[t4] =
                  make_float4(d[4 * t4] + dl[4 * t4], d[4 * t4 + 1] + dl[4 * t4 + 1], d[4 * t4 + 2] + dl[4 * t4 + 2],
                              d[4 * t4 + 3] + dl[4 * t4 + 3]);
          }
          const float sc = sb_scale(sbw[gg]);
#pragma unroll
          for (int t = 0; t < kTPT; t += 2) {
            fma2(y[t], y[t + 1], sc, sc, d[t], d[t + 1]);
            fma2(y[t], y[t + 1], sc, sc, dl[t], dl[t + 1]);
          }
        }
        fence_before();
        mbar_arrive(g_empty + 8 * gb);
        epi_sync<kQEpi>();
#pragma unroll
        for (int gg = 0; gg < kQSG; ++gg) {
          if (gg >= ng) break;
          const float bc = fmaf(-128.0f, sb_scale(sbw[gg]), sb_bias(sbw[gg]));
          const float4* sxv = reinterpret_cast<const float4*>(sx + gg * kQT);
#pragma unroll
          for (int t4 = 0; t4 < kTPT / 4; ++t4) {
            const float4 xv = sxv[t4];
            fma2(y[4 * t4], y[4 * t4 + 1], bc, bc, xv.x, xv.y);
            fma2(y[4 * t4 + 2], y[4 * t4 + 3], bc, bc, xv.z, xv.w);
          }
        }
#pragma unroll
        for (int gg = 0; gg < kQSG; ++gg) sbw[gg] = sbn[gg];
        if (pend_tile >= 0 && (js == kQDefer || js == spu - 1)) finish_pending();
      }
      const bool live = ok && row_ok;
      if (p.S > 1) {
        tcdec::split_write<kTPT>(p, y, kTPT * c, n, split, live);
        pend_tile = tile;
        pend_n = n;
        pend_live = live;
      } else {
        tcdec::fused_epilogue<IN, EPI, kTPT>(p, y, kTPT * c, n, live, lane, s_inv, s_best);
      }
    }
    if (pend_tile >= 0) finish_pending();
    if constexpr (EPI == kEpiLmHead) {
      epi_sync<kQEpi>();
      if (et < p.M && s_best[et] != 0ull) atomicMax(p.amax_key + et, s_best[et]);
    }
  }
  griddep_launch_dependents();
  fence_before();
  __syncthreads();
  tl_mark(p.tl, 2);
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kQTmemCols) : "memory");
  if (!ok && p.status) atomicOr(p.status, kStatusTimeout);
  if constexpr (EPI == kEpiLmHead) {  // the last CTA publishes every token's argmax
    __threadfence();
    if (tid == 0) *s_ticket = atomicAdd(&p.counters[n_tiles], 1u);
    __syncthreads();
    if (*s_ticket == gridDim.x - 1) {
      __threadfence();
      for (int b = tid; b < p.M; b += kQThreads) p.argmax_out[b] = argmax_key_index(atomicOr(p.amax_key + b, 0ull));
      if (tid == 0) p.counters[n_tiles] = 0u;
    }
  }
}

namespace {

using EncodeTiledQ = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledQ encoder_q() {
  static EncodeTiledQ fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledQ>(ptr);
  }
  return fn;
}

template <int IN, int EPI>
cudaError_t launch_q4tc_t(const LaunchCtx& c, const CUtensorMap& mx, const CUtensorMap& mc, const Q4tcParams& p,
                          bool prepare) {
  if (prepare)
    return cudaFuncSetAttribute(k_gemm_q4tc<IN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
  const int units = ((p.N + kQRows - 1) / kQRows) * p.S;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units < p.ctas ? units : p.ctas));
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = kQSmem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemm_q4tc<IN, EPI>, mx, mc, p);
}

cudaError_t dispatch_q4tc(const LaunchCtx& c, const CUtensorMap& mx, const CUtensorMap& mc, const Q4tcParams& p,
                          int in_mode, int epi, bool prepare) {
  if (in_mode == kInNorm && epi == kEpiStore) return launch_q4tc_t<kInNorm, kEpiStore>(c, mx, mc, p, prepare);
  if (in_mode == kInPlain && epi == kEpiStore) return launch_q4tc_t<kInPlain, kEpiStore>(c, mx, mc, p, prepare);
  if (in_mode == kInPlain && epi == kEpiResid) return launch_q4tc_t<kInPlain, kEpiResid>(c, mx, mc, p, prepare);
  if (in_mode == kInNorm && epi == kEpiSwiglu) return launch_q4tc_t<kInNorm, kEpiSwiglu>(c, mx, mc, p, prepare);
  if (in_mode == kInNorm && epi == kEpiLmHead) return launch_q4tc_t<kInNorm, kEpiLmHead>(c, mx, mc, p, prepare);
  return cudaErrorInvalidValue;
}

}  // namespace

int q4tc_max_tokens() { return kQT; }

// K splits of an N x K projection: a divisor of the K / 64 groups (at most 8) that brings the
// units of the one-CTA-per-SM grid closest to whole waves; a larger split count only when it
// gains 10% of the waves' occupancy (each split adds a partial round trip, and short units
// pay their epilogue more often: 8 splits of the 8B gate/up were the slowest measured)
int q4tc_splits(int N, int K, int num_sms) {
  const int tiles = (N + kQRows - 1) / kQRows, groups = K / kQK;
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= 8 && s <= groups; ++s) {
    if (groups % s) continue;
    const long long units = static_cast<long long>(tiles) * s;
    const long long waves = (units + num_sms - 1) / num_sms;
    const double eff = static_cast<double>(units) / static_cast<double>(waves * num_sms);
    if (eff > best_eff + 0.10) {
      best = s;
      best_eff = eff;
    }
  }
  return best;
}

// 4-bit codes [N][K/2] bytes, boxes of 64 bytes x 120 rows (two groups of a tile), no swizzle;
// rows past the end read as zero
cudaError_t q4tc_code_map(void* map128, const void* codes, int N, int K) {
  EncodeTiledQ enc = encoder_q();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kQCodeRow), static_cast<cuuint32_t>(kQRows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(static_cast<CUtensorMap*>(map128), CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes),
                         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gemm_q4tc(const LaunchCtx& c, const void* map_x, const void* map_codes, const Q4tcParams& p,
                             int in_mode, int epi) {
  return dispatch_q4tc(c, *static_cast<const CUtensorMap*>(map_x), *static_cast<const CUtensorMap*>(map_codes), p,
                       in_mode, epi, false);
}

cudaError_t prepare_gemm_q4tc(int in_mode, int epi) {
  CUtensorMap dummy{};
  Q4tcParams p{};
  return dispatch_q4tc(LaunchCtx{nullptr, false}, dummy, dummy, p, in_mode, epi, true);
}

}  // namespace dec

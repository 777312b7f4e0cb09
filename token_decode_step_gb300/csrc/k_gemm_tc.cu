// Batched (B >= 2) fused projections on tensor cores: Y[b][n] = sum_k W[n][k] X[b][k]
// with mma.sync m16n8k16 (weights as the 16-row A operand, tokens as the 8-column
// B operand, fp32 accumulation), RMSNorm folded into the X staging and the same
// epilogues as the batch-1 GEMV (store / residual + sum of squares / SwiGLU /
// lm_head argmax).
//
// Sources: Butter architecture.md "SINGLE-TOKEN DECODE" (the gemv sequence);
// oxinfer crate page "MLX checkpoints" (affine 4-bit, w = scale*q + bias, the
// per-group sum-of-x factoring); oxinfer's batched decode notes (a batch of
// sequences reads the weights once).  With B sequences the projection is a
// small dense contraction (B x K times K x N), so it runs on the tensor pipe.
//
// Weight layout (packed at create time, see k_misc.cu):
//   bf16: tiles of 16 rows x 16 inputs, 512 bytes, lane-major: lane (g = lane/4,
//         t = lane%4) holds its four A registers (rows g and g+8, inputs 2t, 2t+1
//         and 2t+8, 2t+9) in 16 contiguous bytes, so a warp reads a tile with one
//         coalesced 16-byte load per lane and needs no shuffles.
//   4-bit: tiles of 16 rows x 64 inputs (one quantisation group), 576 bytes:
//         512 bytes of codes (lane-major, one 32-bit word per 16-input k-step,
//         arranged so that (word >> 4i) & 0x000F000F yields A register i), then
//         for each g the bf16 (scale, bias) of rows g and g+8.
// Activations: staged in shared memory as bf16 hi + lo rows (x = hi + lo, ~16
// significant bits; one row per token and half, padded by 16 bytes to keep
// ldmatrix conflict-free), so every 8 tokens take two n-tiles.  bf16 weights are
// the A operand as they are; 4-bit weights enter as their exact integer codes q
// (bf16), and the group scale and bias are applied in fp32 after each group:
// y += s * sum(q x) + b * sum(x).
#include <cuda_fp16.h>

#include "dec_internal.cuh"
#include "q4.cuh"

namespace dec {

namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t smem_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1]) : "r"(smem_addr));
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

}  // namespace

size_t gemm_tc_smem_bytes(int wfmt, int ny, int kc) {
  const int nt = 2 * ny;
  size_t b = static_cast<size_t>(nt) * 8 * (kc + 8) * 2;
  if (wfmt == kWQ4) b += static_cast<size_t>(kc / kGroup) * ny * 8 * 4;
  return b;
}

template <int WF, int NY, int TPW, int IN, int EPI>
__global__ void __launch_bounds__(kWarps * 32) k_gemm_tc(GemmParams p) {
  constexpr int NT = 2 * NY;  // n-tiles of the MMA: hi rows of every token, then lo rows
  constexpr int XR = NT * 8;              // staged activation rows
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float s_inv[32];
  __shared__ unsigned s_ticket;

  const int KC = p.KC, KSP = p.KC + 8;  // staged chunk of the split, padded rows
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  float* xsum = reinterpret_cast<float*>(smem + static_cast<size_t>(XR) * KSP * 2);  // [KS/64][NY*8]

  const int rb = blockIdx.x, split = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
  const int kbeg0 = split * p.KS;
  const int n_rt = p.Npad / 16;
  const int rt0 = (rb * kWarps + warp) * TPW;

  griddep_wait();

  // ---- per-token inverse RMS (fused RMSNorm), then stage X for this K split
  if constexpr (IN == kInNorm) {
    for (int b = warp; b < p.B; b += kWarps) {
      float s = 0.f;
      for (int i = lane; i < p.n_sumsq_in; i += 32) s += p.sumsq_in[static_cast<size_t>(b) * p.n_sumsq_in + i];
      s = warp_sum(s);
      if (lane == 0) s_inv[b] = rsqrtf(s / static_cast<float>(p.K) + p.eps);
    }
  }
  // ---- main loop: each warp owns TPW row tiles over the whole K split, staged chunk by chunk
  float acc[TPW][NT][4];
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[i][n][0] = acc[i][n][1] = acc[i][n][2] = acc[i][n][3] = 0.f;
  bool valid[TPW];
#pragma unroll
  for (int i = 0; i < TPW; ++i) valid[i] = (rt0 + i) < n_rt;

  {  // rows of absent tokens (and their lo rows) stay zero for every chunk
    uint4* z = reinterpret_cast<uint4*>(smem);
    const int nz = XR * KSP * 2 / 16;
    for (int i = tid; i < nz; i += kWarps * 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  for (int kbeg = kbeg0; kbeg < kbeg0 + p.KS; kbeg += KC) {
    if (kbeg != kbeg0) __syncthreads();  // previous chunk fully consumed
    const int k4 = KC / 4;
    for (int idx = tid; idx < p.B * k4; idx += kWarps * 32) {
      const int b = idx / k4, kq = idx % k4;
      const int col = kbeg + 4 * kq;
      float4 v = *reinterpret_cast<const float4*>(p.x + static_cast<size_t>(b) * p.K + col);
      if constexpr (IN == kInNorm) {
        const uint2 wn = *reinterpret_cast<const uint2*>(p.norm_w + col);
        const float r = s_inv[b];
        v.x = (v.x * r) * bf16_lo(wn.x);
        v.y = (v.y * r) * bf16_hi(wn.x);
        v.z = (v.z * r) * bf16_lo(wn.y);
        v.w = (v.w * r) * bf16_hi(wn.y);
      }
      uint16_t* dst = xs + static_cast<size_t>(b) * KSP + 4 * kq;
      const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y), h23 = __floats2bfloat162_rn(v.z, v.w);
      const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
      const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
      const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
      uint2 hv, lv;
      hv.x = *reinterpret_cast<const uint32_t*>(&h01);
      hv.y = *reinterpret_cast<const uint32_t*>(&h23);
      lv.x = *reinterpret_cast<const uint32_t*>(&l01);
      lv.y = *reinterpret_cast<const uint32_t*>(&l23);
      *reinterpret_cast<uint2*>(dst) = hv;
      *reinterpret_cast<uint2*>(dst + static_cast<size_t>(NY) * 8 * KSP) = lv;
    }
    __syncthreads();
    if constexpr (WF == kWQ4) {
      // per (group, token) sum of the staged inputs (hi + lo), for the bias term: together
      // with the MMA over the same staged values this is sum_k (s q_k + b) x_k
      const int ng = KC / kGroup;
      for (int idx = tid; idx < ng * NY * 8; idx += kWarps * 32) {
        const int grp = idx / (NY * 8), b = idx % (NY * 8);
        const __nv_bfloat16* hi = reinterpret_cast<const __nv_bfloat16*>(xs) + static_cast<size_t>(b) * KSP + grp * kGroup;
        const __nv_bfloat16* lo = hi + static_cast<size_t>(NY) * 8 * KSP;
        float s = 0.f;
#pragma unroll 8
        for (int i = 0; i < kGroup; ++i) s += __bfloat162float(hi[i]) + __bfloat162float(lo[i]);
        xsum[idx] = s;
      }
      __syncthreads();
    }
    const uint32_t xs_base = smem_u32(xs);
    // ldmatrix lane address for n-tile pair np at input column c (within the split)
    auto b_frags = [&](int c, uint32_t (&bf)[NT][2]) {
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        const int row = (2 * np + (mi >> 1)) * 8 + rr;
        uint32_t r[4];
        ldmatrix_x4(r, xs_base + (row * KSP + c + 8 * (mi & 1)) * 2);
        bf[2 * np][0] = r[0];
        bf[2 * np][1] = r[1];
        bf[2 * np + 1][0] = r[2];
        bf[2 * np + 1][1] = r[3];
      }
      if constexpr (NT % 2 == 1) {
        const int row = (NT - 1) * 8 + rr;
        uint32_t r[2];
        ldmatrix_x2(r, xs_base + (row * KSP + c + 8 * ((lane >> 3) & 1)) * 2);
        bf[NT - 1][0] = r[0];
        bf[NT - 1][1] = r[1];
      }
    };

    if constexpr (WF == kWBf16) {
      const int nk = KC / 16, kt0 = kbeg / 16, ktiles = p.K / 16;
      const uint4* wbase = static_cast<const uint4*>(p.w);
      for (int kk = 0; kk < nk; kk += 4) {
        uint4 a[TPW][4];
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            a[i][u] = valid[i] ? ld_stream16(wbase + (static_cast<size_t>(rt0 + i) * ktiles + kt0 + kk + u) * 32 + lane)
                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t bf[NT][2];
          b_frags((kk + u) * 16, bf);
#pragma unroll
          for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int n = 0; n < NT; ++n)
              mma_bf16_16816(acc[i][n], a[i][u].x, a[i][u].y, a[i][u].z, a[i][u].w, bf[n][0], bf[n][1]);
        }
      }
    } else {
      const int ngrp = KC / kGroup, g0 = kbeg / kGroup, gtiles = p.K / kGroup;
      const unsigned char* wbase = static_cast<const unsigned char*>(p.w);
      for (int grp = 0; grp < ngrp; ++grp) {
        uint4 nib[TPW];
        uint2 sbv[TPW];
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          const unsigned char* tile = wbase + (static_cast<size_t>(rt0 + i) * gtiles + g0 + grp) * 576;
          nib[i] = valid[i] ? ld_stream16(tile + lane * 16) : make_uint4(0u, 0u, 0u, 0u);
          sbv[i] = valid[i] ? __ldg(reinterpret_cast<const uint2*>(tile + 512 + g * 8)) : make_uint2(0u, 0u);
        }
        float gacc[TPW][NT][4];
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
          for (int n = 0; n < NT; ++n) gacc[i][n][0] = gacc[i][n][1] = gacc[i][n][2] = gacc[i][n][3] = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t bf[NT][2];
          b_frags(grp * kGroup + u * 16, bf);
#pragma unroll
          for (int i = 0; i < TPW; ++i) {
            const uint32_t word = u == 0 ? nib[i].x : u == 1 ? nib[i].y : u == 2 ? nib[i].z : nib[i].w;
            const uint32_t a0 = q4_pair_bf16(word, 0), a1 = q4_pair_bf16(word, 4);
            const uint32_t a2 = q4_pair_bf16(word, 8), a3 = q4_pair_bf16(word, 12);
#pragma unroll
            for (int n = 0; n < NT; ++n) mma_bf16_16816(gacc[i][n], a0, a1, a2, a3, bf[n][0], bf[n][1]);
          }
        }
        const float* xg = xsum + grp * NY * 8;
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          const float s_lo = bf16_lo(sbv[i].x), b_lo = bf16_hi(sbv[i].x);  // row g
          const float s_hi = bf16_lo(sbv[i].y), b_hi = bf16_hi(sbv[i].y);  // row g + 8
#pragma unroll
          for (int n = 0; n < NY; ++n)  // hi n-tile n and lo n-tile n + NY hold the same tokens
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float xs_e = xg[8 * n + 2 * t + (e & 1)];
              const float sc = (e < 2) ? s_lo : s_hi, bi = (e < 2) ? b_lo : b_hi;
              acc[i][n][e] = fmaf(sc, gacc[i][n][e] + gacc[i][n + NY][e], fmaf(bi, xs_e, acc[i][n][e]));
            }
        }
      }
    }
  }
  griddep_launch_dependents();

  // ---- y[i][n][e]: row 16 rt + g + 8 (e >> 1), token 8 n + 2 t + (e & 1)
  float y[TPW][NY][4];
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int n = 0; n < NY; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) y[i][n][e] = (WF == kWBf16) ? acc[i][n][e] + acc[i][n + NY][e] : acc[i][n][e];

  // ---- split-K: the last CTA of a row block adds the S partials in split order
  if (p.S > 1) {
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      if (!valid[i]) continue;
      float* dst = p.partials + ((static_cast<size_t>(split) * n_rt + rt0 + i) * 32 + lane) * (NY * 4);
#pragma unroll
      for (int n = 0; n < NY; ++n)
        *reinterpret_cast<float4*>(dst + 4 * n) = make_float4(y[i][n][0], y[i][n][1], y[i][n][2], y[i][n][3]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_ticket = atomicAdd(&p.counters[rb], 1u);
    __syncthreads();
    if (s_ticket != static_cast<unsigned>(p.S - 1)) return;
    __threadfence();
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      if (!valid[i]) continue;
#pragma unroll
      for (int n = 0; n < NY; ++n) y[i][n][0] = y[i][n][1] = y[i][n][2] = y[i][n][3] = 0.f;
      for (int s = 0; s < p.S; ++s) {
        const float* src = p.partials + ((static_cast<size_t>(s) * n_rt + rt0 + i) * 32 + lane) * (NY * 4);
#pragma unroll
        for (int n = 0; n < NY; ++n) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + 4 * n));
          y[i][n][0] += v.x;
          y[i][n][1] += v.y;
          y[i][n][2] += v.z;
          y[i][n][3] += v.w;
        }
      }
    }
    if (tid == 0) p.counters[rb] = 0u;
  }

  // ---- epilogue
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    if (!valid[i]) continue;
    const int rt = rt0 + i;
#pragma unroll
    for (int n = 0; n < NY; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 16 * rt + g + 8 * (e >> 1);
        const int tok = 8 * n + 2 * t + (e & 1);
        if constexpr (EPI == kEpiStore) {
          if (row < p.N && tok < p.B) p.out[static_cast<size_t>(tok) * p.N + row] = y[i][n][e];
        } else if constexpr (EPI == kEpiResid) {
          float hn = 0.f;
          if (tok < p.B) {
            float* hp = p.out + static_cast<size_t>(tok) * p.N + row;
            hn = *hp + y[i][n][e];
            *hp = hn;
          }
          float ss = hn * hn;  // sum over the 8 rows g of this half-tile (lanes with equal t)
          ss += __shfl_xor_sync(0xffffffffu, ss, 4);
          ss += __shfl_xor_sync(0xffffffffu, ss, 8);
          ss += __shfl_xor_sync(0xffffffffu, ss, 16);
          if (g == 0 && tok < p.B) p.sumsq_out[static_cast<size_t>(tok) * (p.N / kResGroup) + 2 * rt + (e >> 1)] = ss;
        } else if constexpr (EPI == kEpiSwiglu) {
          // rows 0..7 of a tile are gate rows, rows 8..15 the matching up rows
          if (e < 2 && tok < p.B)
            p.out[static_cast<size_t>(tok) * (p.N / 2) + 8 * rt + g] = silu_f(y[i][n][e]) * y[i][n][e + 2];
        } else {  // lm_head
          if (row < p.N && tok < p.B && p.out) p.out[static_cast<size_t>(tok) * p.N + row] = y[i][n][e];
        }
      }
      if constexpr (EPI == kEpiLmHead) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // token 8 n + 2 t + c: rows g (e = c) and g + 8 (e = c + 2)
          const int r0 = 16 * rt + g, r1 = r0 + 8;
          unsigned long long k0 = r0 < p.N ? argmax_key(y[i][n][c], r0) : 0ull;
          unsigned long long k1 = r1 < p.N ? argmax_key(y[i][n][c + 2], r1) : 0ull;
          unsigned long long k = k0 > k1 ? k0 : k1;
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, k, o);
            k = other > k ? other : k;
          }
          const int tok = 8 * n + 2 * t + c;
          if (g == 0 && tok < p.B) atomicMax(p.amax_key + tok, k);
        }
      }
    }
  }
  if constexpr (EPI == kEpiLmHead) {
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const unsigned nblk = gridDim.x;
      const unsigned done = atomicAdd(&p.counters[nblk], 1u);
      if (done == nblk - 1) {
        __threadfence();
        for (int b = 0; b < p.B; ++b) p.argmax_out[b] = argmax_key_index(atomicOr(p.amax_key + b, 0ull));
        p.counters[nblk] = 0u;
      }
    }
  }
}

namespace {

template <int WF, int NY, int TPW, int IN, int EPI>
cudaError_t launch_t(const LaunchCtx& c, const GemmParams& p, bool prepare) {
  auto kern = k_gemm_tc<WF, NY, TPW, IN, EPI>;
  const size_t smem = gemm_tc_smem_bytes(WF, NY, p.KC);
  if (prepare) return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  const int n_rt = p.Npad / 16;
  const int per_blk = kWarps * TPW;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n_rt + per_blk - 1) / per_blk, p.S);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int WF, int NY, int TPW>
cudaError_t dispatch_epi(const LaunchCtx& c, const GemmParams& p, int in_mode, int epi, bool prepare) {
  if (in_mode == kInNorm && epi == kEpiStore) return launch_t<WF, NY, TPW, kInNorm, kEpiStore>(c, p, prepare);
  if (in_mode == kInPlain && epi == kEpiResid) return launch_t<WF, NY, TPW, kInPlain, kEpiResid>(c, p, prepare);
  if (in_mode == kInNorm && epi == kEpiSwiglu) return launch_t<WF, NY, TPW, kInNorm, kEpiSwiglu>(c, p, prepare);
  if (in_mode == kInNorm && epi == kEpiLmHead) return launch_t<WF, NY, TPW, kInNorm, kEpiLmHead>(c, p, prepare);
  return cudaErrorInvalidValue;
}

cudaError_t dispatch(const LaunchCtx& c, const GemmParams& p, int wfmt, int in_mode, int epi, bool prepare) {
  const int ny = gemm_tc_ny(wfmt, p.B);
  if (wfmt == kWBf16) {
    if (ny == 1) return dispatch_epi<kWBf16, 1, 1>(c, p, in_mode, epi, prepare);
    if (ny == 2) return dispatch_epi<kWBf16, 2, 1>(c, p, in_mode, epi, prepare);
  } else {
    if (ny == 1) return dispatch_epi<kWQ4, 1, 2>(c, p, in_mode, epi, prepare);
    if (ny == 2) return dispatch_epi<kWQ4, 2, 2>(c, p, in_mode, epi, prepare);
    if (ny == 4) return dispatch_epi<kWQ4, 4, 1>(c, p, in_mode, epi, prepare);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int gemm_tc_ny(int wfmt, int batch) {
  const int ny = (batch + 7) / 8;
  if (wfmt == kWBf16) return ny <= 2 ? ny : 0;
  return ny <= 1 ? 1 : ny <= 2 ? 2 : ny <= 4 ? 4 : 0;
}

int gemm_tc_rows_per_block(int wfmt, int ny) { return kWarps * 16 * (wfmt == kWQ4 && ny <= 2 ? 2 : 1); }

cudaError_t launch_gemm_tc(const LaunchCtx& c, const GemmParams& p, int wfmt, int in_mode, int epi) {
  return dispatch(c, p, wfmt, in_mode, epi, false);
}

cudaError_t prepare_gemm_tc(const GemmParams& p, int wfmt, int in_mode, int epi) {
  return dispatch(LaunchCtx{nullptr, false}, p, wfmt, in_mode, epi, true);
}

}  // namespace dec

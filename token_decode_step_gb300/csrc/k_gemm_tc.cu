// Batched (B >= 2) fused projections on tensor cores: Y[b][n] = sum_k W[n][k] X[b][k]
// with mma.sync m16n8k16 (weights as the 16-row A operand, tokens as the 8-column
// B operand, fp32 accumulation) and the same fused steps as the batch-1 GEMV:
// RMSNorm of the input, then store / residual add + sum of squares / SwiGLU /
// lm_head argmax.
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
// Activations: the producing kernel already wrote them as bf16 hi + lo planes
// ([2][B][K], x = hi + lo, ~16 significant bits), for norm inputs multiplied by
// the norm weight; the per-token 1/rms is applied to the products afterwards
// (the product is linear in x).  Chunks of KC inputs are copied into shared
// memory with cp.async, double-buffered, one padded row per token and half
// (16-byte padding keeps ldmatrix conflict-free), so every 8 tokens take two
// n-tiles.  4-bit weights enter as exact integer codes q (bf16) and the group
// scale and bias are applied in fp32 after each group: y += s*sum(q x) + b*sum(x).
#include <type_traits>

#include "dec_internal.cuh"
#include "q4.cuh"

namespace dec {

namespace {

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// (hi, lo) bf16 split of a float: hi = bf16(v), lo = bf16(v - hi)
__device__ __forceinline__ void split_hl(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

}  // namespace

size_t gemm_tc_smem_bytes(int wfmt, int ny, int kc) {
  size_t b = 2ull * (2 * ny * 8) * (kc + 8) * 2;              // two chunk buffers
  if (wfmt == kWQ4) b += 2ull * (kc / kGroup) * ny * 8 * 4;  // two group-sum buffers
  return b;
}

template <int WF, int NY, int TPW, int WARPS, int IN, int EPI>
__global__ void __launch_bounds__(WARPS * 32, WARPS == 8 ? 2 : 1) k_gemm_tc(GemmParams p) {
  constexpr int NT = 2 * NY;  // n-tiles of the MMA: hi rows of every token, then lo rows
  constexpr int XR = NT * 8;  // staged rows per chunk buffer
  constexpr int NTH = WARPS * 32;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float s_inv[32];
  __shared__ unsigned s_ticket;

  const int KC = p.KC, KSP = p.KC + 8;  // staged chunk, padded row length
  const size_t buf_elems = static_cast<size_t>(XR) * KSP;
  uint16_t* xs0 = reinterpret_cast<uint16_t*>(smem);
  float* xsum0 = reinterpret_cast<float*>(smem + 2 * buf_elems * 2);  // two [KC/64][NY*8] buffers

  // x = row block * tblocks + token block (token blocks vary fastest, so that the CTAs
  // streaming one weight tile for the different token blocks run together and all but
  // the first read it from L2); y = K split (a single split when tblocks > 1)
  const int tb = blockIdx.x % p.tblocks, rb = blockIdx.x / p.tblocks, split = blockIdx.y;
  const int tok0 = tb * NY * 8;                                  // this block's first token
  const int nb = p.B - tok0 < NY * 8 ? p.B - tok0 : NY * 8;      // and its number of tokens
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
  const int kbeg0 = split * p.KS;
  const int n_rt = p.Npad / 16;
  const int rt0 = (rb * WARPS + warp) * TPW;
  const int nchunks = p.KS / KC;

  bool valid[TPW];
#pragma unroll
  for (int i = 0; i < TPW; ++i) valid[i] = (rt0 + i) < n_rt;

  tl_mark(p.tl, 0);
  {  // rows of absent tokens (and their lo rows) stay zero in both buffers
    uint4* z = reinterpret_cast<uint4*>(smem);
    const int nz = static_cast<int>(2 * buf_elems * 2 / 16);
    for (int i = tid; i < nz; i += NTH) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }

  // The K split is walked in units of 64 inputs (4 bf16 k-tiles, or one 4-bit group);
  // each lane keeps the weights of PF units in flight in a register ring, across the
  // chunk boundaries of the staged activations.
  constexpr int PF = kGemmPrefetch;
  using Unit = typename std::conditional<WF == kWBf16, uint4[TPW][4], uint4[TPW][2]>::type;
  const int nunits = p.KS / 64, upc = KC / 64;
  const int ktiles = p.K / 16, gtiles = p.K / kGroup;
  auto load_unit = [&](int u, Unit& dst) {
    const int ug = kbeg0 / 64 + u;  // 64-input unit index along the whole K
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      if constexpr (WF == kWBf16) {
        const uint4* wb = static_cast<const uint4*>(p.w) + (static_cast<size_t>(rt0 + i) * ktiles + 4 * ug) * 32 + lane;
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[i][q] = valid[i] ? ld_stream16(wb + q * 32) : make_uint4(0u, 0u, 0u, 0u);
      } else {
        const unsigned char* tile = static_cast<const unsigned char*>(p.w) + (static_cast<size_t>(rt0 + i) * gtiles + ug) * 576;
        dst[i][0] = valid[i] ? ld_stream16(tile + lane * 16) : make_uint4(0u, 0u, 0u, 0u);
        const uint2 sb = valid[i] ? __ldg(reinterpret_cast<const uint2*>(tile + 512 + g * 8)) : make_uint2(0u, 0u);
        dst[i][1] = make_uint4(sb.x, sb.y, 0u, 0u);
      }
    }
  };
  // weights do not depend on upstream kernels: the first PF units are requested
  // before the grid-dependency wait
  Unit ring[PF];
#pragma unroll
  for (int j = 0; j < PF; ++j)
    if (j < nunits) load_unit(j, ring[j]);
  // Residual epilogue inputs: the residual rows (last written two or more kernels
  // upstream, which completed before the previous kernel could pass its own wait and
  // start this one) and the next norm's weights, requested before the wait too.
  constexpr int RH = EPI == kEpiResid ? 1 : 0;
  float h_pre[RH ? TPW : 1][RH ? NY : 1][4];
  float nw_pre[RH ? TPW : 1][2];
  if constexpr (RH) {
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int row = 16 * (rt0 + i) + g + 8 * hf;
        nw_pre[i][hf] = (valid[i] && row < p.N) ? bf16_to_f(p.next_norm_w[row]) : 0.f;
      }
#pragma unroll
      for (int n = 0; n < NY; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = 16 * (rt0 + i) + g + 8 * (e >> 1), tok = 8 * n + 2 * t + (e & 1);
          h_pre[i][n][e] = (valid[i] && row < p.N && tok < nb)
                               ? __ldcg(p.out + static_cast<size_t>(tok0 + tok) * p.N + row)
                               : 0.f;
        }
    }
  }

  griddep_wait();
  tl_mark(p.tl, 1);

  if constexpr (IN == kInNorm) {  // per-token 1/rms of the residual (fused RMSNorm)
    for (int b = warp; b < nb; b += WARPS) {
      float s = 0.f;
      for (int i = lane; i < p.n_sumsq_in; i += 32) s += p.sumsq_in[static_cast<size_t>(tok0 + b) * p.n_sumsq_in + i];
      s = warp_sum(s);
      if (lane == 0) s_inv[b] = rsqrtf(s / static_cast<float>(p.K) + p.eps);
    }
  }
  __syncthreads();

  // copy chunk c (inputs kbeg0 + c KC ..) of both planes into buffer c & 1
  auto issue_chunk = [&](int c) {
    const uint32_t dst0 = smem_u32(xs0 + (c & 1) * buf_elems);
    const int per_row = KC / 8;  // 16-byte pieces
    const int kb = kbeg0 + c * KC;
    for (int idx = tid; idx < 2 * nb * per_row; idx += NTH) {
      const int r = idx / per_row, j = idx % per_row;
      const int plane = r / nb, b = r % nb;
      const __nv_bfloat16* src = p.xhl + (static_cast<size_t>(plane) * p.B + tok0 + b) * p.K + kb + 8 * j;
      const int srow = plane * NY * 8 + b;
      cp_async16(dst0 + (srow * KSP + 8 * j) * 2, src, 16);
    }
    cp_async_commit();
  };

  float acc[TPW][NT][4];
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[i][n][0] = acc[i][n][1] = acc[i][n][2] = acc[i][n][3] = 0.f;

  issue_chunk(0);
  const uint16_t* xs = xs0;
  float* xsum = xsum0;
  uint32_t xs_base = smem_u32(xs0);
  // ldmatrix: B fragments of every n-tile at input column cc (within the chunk)
  auto b_frags = [&](int cc, uint32_t (&bf)[NT][2]) {
    const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      const int row = (2 * np + (mi >> 1)) * 8 + rr;
      uint32_t r[4];
      ldmatrix_x4(r, xs_base + (row * KSP + cc + 8 * (mi & 1)) * 2);
      bf[2 * np][0] = r[0];
      bf[2 * np][1] = r[1];
      bf[2 * np + 1][0] = r[2];
      bf[2 * np + 1][1] = r[3];
    }
  };

  for (int u0 = 0; u0 < nunits; u0 += PF) {
#pragma unroll
    for (int j = 0; j < PF; ++j) {
      const int u = u0 + j;
      if (u >= nunits) break;
      const int c = u / upc, uc = u % upc;  // chunk and unit within it
      if (uc == 0) {  // activations of chunk c: wait for them, prefetch chunk c + 1
        if (c + 1 < nchunks) {
          issue_chunk(c + 1);
          cp_async_wait<1>();
        } else {
          cp_async_wait<0>();
        }
        __syncthreads();
        xs = xs0 + (c & 1) * buf_elems;
        xs_base = smem_u32(xs);
        xsum = xsum0 + (c & 1) * (KC / kGroup) * NY * 8;
        if constexpr (WF == kWQ4) {
          // per (group, token) sum of the staged inputs (hi + lo), for the bias term: with
          // the MMA over the same staged values this is sum_k (s q_k + b) x_k
          const int ng = KC / kGroup;
          for (int idx = tid; idx < ng * NY * 8; idx += NTH) {
            const int grp = idx / (NY * 8), b = idx % (NY * 8);
            const uint4* hi = reinterpret_cast<const uint4*>(xs + static_cast<size_t>(b) * KSP + grp * kGroup);
            const uint4* lo = reinterpret_cast<const uint4*>(xs + static_cast<size_t>(NY * 8 + b) * KSP + grp * kGroup);
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < kGroup / 8; ++q) {
              const uint4 va = hi[q], vd = lo[q];
              sum += (bf16_lo(va.x) + bf16_hi(va.x)) + (bf16_lo(va.y) + bf16_hi(va.y)) +
                     (bf16_lo(va.z) + bf16_hi(va.z)) + (bf16_lo(va.w) + bf16_hi(va.w));
              sum += (bf16_lo(vd.x) + bf16_hi(vd.x)) + (bf16_lo(vd.y) + bf16_hi(vd.y)) +
                     (bf16_lo(vd.z) + bf16_hi(vd.z)) + (bf16_lo(vd.w) + bf16_hi(vd.w));
            }
            xsum[idx] = sum;
          }
          __syncthreads();
        }
      }

      if constexpr (WF == kWBf16) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t bf[NT][2];
          b_frags(uc * 64 + q * 16, bf);
#pragma unroll
          for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int n = 0; n < NT; ++n)
              mma_bf16_16816(acc[i][n], ring[j][i][q].x, ring[j][i][q].y, ring[j][i][q].z, ring[j][i][q].w, bf[n][0],
                             bf[n][1]);
        }
      } else {
        float gacc[TPW][NT][4];
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
          for (int n = 0; n < NT; ++n) gacc[i][n][0] = gacc[i][n][1] = gacc[i][n][2] = gacc[i][n][3] = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t bf[NT][2];
          b_frags(uc * kGroup + q * 16, bf);
#pragma unroll
          for (int i = 0; i < TPW; ++i) {
            const uint4 nib = ring[j][i][0];
            const uint32_t word = q == 0 ? nib.x : q == 1 ? nib.y : q == 2 ? nib.z : nib.w;
            const uint32_t a0 = q4_pair_bf16(word, 0), a1 = q4_pair_bf16(word, 4);
            const uint32_t a2 = q4_pair_bf16(word, 8), a3 = q4_pair_bf16(word, 12);
#pragma unroll
            for (int n = 0; n < NT; ++n) mma_bf16_16816(gacc[i][n], a0, a1, a2, a3, bf[n][0], bf[n][1]);
          }
        }
        const float* xg = xsum + uc * NY * 8;
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          const uint4 sb = ring[j][i][1];
          const float s_lo = bf16_lo(sb.x), b_lo = bf16_hi(sb.x);  // row g
          const float s_hi = bf16_lo(sb.y), b_hi = bf16_hi(sb.y);  // row g + 8
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
      if (u + PF < nunits) load_unit(u + PF, ring[j]);  // refill the slot just consumed
      if (uc == upc - 1) __syncthreads();               // buffer c & 1 is refilled with chunk c + 2
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
    if (s_ticket != static_cast<unsigned>(p.S - 1)) {
      tl_mark(p.tl, 2);
      return;
    }
    __threadfence();
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      if (!valid[i]) continue;
#pragma unroll
      for (int n = 0; n < NY; ++n) y[i][n][0] = y[i][n][1] = y[i][n][2] = y[i][n][3] = 0.f;
      // four splits' partials requested at a time, then added in split order
      for (int s0 = 0; s0 < p.S; s0 += 4) {
        float4 v[4][NY];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (s0 + j >= p.S) break;
          const float* src = p.partials + ((static_cast<size_t>(s0 + j) * n_rt + rt0 + i) * 32 + lane) * (NY * 4);
#pragma unroll
          for (int n = 0; n < NY; ++n) v[j][n] = __ldcg(reinterpret_cast<const float4*>(src + 4 * n));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (s0 + j >= p.S) break;
#pragma unroll
          for (int n = 0; n < NY; ++n) {
            y[i][n][0] += v[j][n].x;
            y[i][n][1] += v[j][n].y;
            y[i][n][2] += v[j][n].z;
            y[i][n][3] += v[j][n].w;
          }
        }
      }
    }
    if (tid == 0) p.counters[rb] = 0u;
  }

  if constexpr (IN == kInNorm) {  // the norm's 1/rms, per token
#pragma unroll
    for (int n = 0; n < NY; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = 8 * n + 2 * t + (e & 1);
        const float r = tok < nb ? s_inv[tok] : 0.f;
#pragma unroll
        for (int i = 0; i < TPW; ++i) y[i][n][e] *= r;
      }
  }

  // ---- epilogue
  const size_t plane_out = static_cast<size_t>(p.B) * (EPI == kEpiSwiglu ? p.N / 2 : p.N);
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    if (!valid[i]) continue;
    const int rt = rt0 + i;
#pragma unroll
    for (int n = 0; n < NY; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 16 * rt + g + 8 * (e >> 1);
        const int tok = 8 * n + 2 * t + (e & 1);   // within the block
        const size_t gtok = static_cast<size_t>(tok0 + tok);
        if constexpr (EPI == kEpiStore) {
          if (row < p.N && tok < nb) p.out[gtok * p.N + row] = y[i][n][e];
        } else if constexpr (EPI == kEpiResid) {
          float hn = 0.f;
          if (tok < nb) {
            hn = h_pre[i][n][e] + y[i][n][e];
            p.out[gtok * p.N + row] = hn;
            // the next consumer's input: h times its norm weight, as hi + lo planes
            __nv_bfloat16 hi, lo;
            split_hl(hn * nw_pre[i][e >> 1], hi, lo);
            const size_t o = gtok * p.N + row;
            p.xhl_out[o] = hi;
            p.xhl_out[plane_out + o] = lo;
          }
          float ss = hn * hn;  // sum over the 8 rows g of this half-tile (lanes with equal t)
          ss += __shfl_xor_sync(0xffffffffu, ss, 4);
          ss += __shfl_xor_sync(0xffffffffu, ss, 8);
          ss += __shfl_xor_sync(0xffffffffu, ss, 16);
          if (g == 0 && tok < nb) p.sumsq_out[gtok * (p.N / kResGroup) + 2 * rt + (e >> 1)] = ss;
        } else if constexpr (EPI == kEpiSwiglu) {
          // rows 0..7 of a tile are gate rows, rows 8..15 the matching up rows
          if (e < 2 && tok < nb) {
            const float gv = silu_f(y[i][n][e]) * y[i][n][e + 2];
            const size_t o = gtok * (p.N / 2) + 8 * rt + g;
            p.out[o] = gv;
            __nv_bfloat16 hi, lo;
            split_hl(gv, hi, lo);
            p.xhl_out[o] = hi;
            p.xhl_out[plane_out + o] = lo;
          }
        } else {  // lm_head
          if (row < p.N && tok < nb && p.out) p.out[gtok * p.N + row] = y[i][n][e];
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
          if (g == 0 && tok < nb) atomicMax(p.amax_key + tok0 + tok, k);
        }
      }
    }
  }
  tl_mark(p.tl, 2);
  if constexpr (EPI == kEpiLmHead) {
    __threadfence();
    __syncthreads();
    const unsigned nblk = gridDim.x;
    if (tid == 0) s_ticket = atomicAdd(&p.counters[nblk], 1u);
    __syncthreads();
    if (s_ticket == nblk - 1) {  // the last CTA publishes every token's argmax
      __threadfence();
      for (int b = tid; b < p.B; b += NTH) p.argmax_out[b] = argmax_key_index(atomicOr(p.amax_key + b, 0ull));
      if (tid == 0) p.counters[nblk] = 0u;
    }
  }
}

namespace {

template <int WF, int NY, int TPW, int WARPS, int IN, int EPI>
cudaError_t launch_t(const LaunchCtx& c, const GemmParams& p, bool prepare) {
  auto kern = k_gemm_tc<WF, NY, TPW, WARPS, IN, EPI>;
  const size_t smem = gemm_tc_smem_bytes(WF, NY, p.KC);
  if (prepare) return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  const int n_rt = p.Npad / 16;
  const int per_blk = WARPS * TPW;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n_rt + per_blk - 1) / per_blk * p.tblocks, p.S);
  cfg.blockDim = dim3(WARPS * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int WF, int NY, int TPW, int WARPS>
cudaError_t dispatch_epi(const LaunchCtx& c, const GemmParams& p, int in_mode, int epi, bool prepare) {
  if (in_mode == kInNorm && epi == kEpiStore) return launch_t<WF, NY, TPW, WARPS, kInNorm, kEpiStore>(c, p, prepare);
  if (in_mode == kInPlain && epi == kEpiResid) return launch_t<WF, NY, TPW, WARPS, kInPlain, kEpiResid>(c, p, prepare);
  if (in_mode == kInNorm && epi == kEpiSwiglu) return launch_t<WF, NY, TPW, WARPS, kInNorm, kEpiSwiglu>(c, p, prepare);
  if (in_mode == kInNorm && epi == kEpiLmHead) return launch_t<WF, NY, TPW, WARPS, kInNorm, kEpiLmHead>(c, p, prepare);
  return cudaErrorInvalidValue;
}

// Tile shapes: bf16 - 8 warps of one 16-row tile (128 rows per CTA); 4-bit - 8 warps
// of two tiles up to 16 tokens, 16 warps of one tile for 17..32 tokens (256 rows
// share each staged chunk of activations).
cudaError_t dispatch(const LaunchCtx& c, const GemmParams& p, int wfmt, int in_mode, int epi, bool prepare) {
  if (p.tblocks < 1) return cudaErrorInvalidValue;
  const int ny = gemm_tc_ny(wfmt, p.tblocks > 1 ? gemm_tc_block_tokens(wfmt) : p.B);
  if (wfmt == kWBf16) {
    if (ny == 1) return dispatch_epi<kWBf16, 1, 1, 8>(c, p, in_mode, epi, prepare);
    if (ny == 2) return dispatch_epi<kWBf16, 2, 1, 8>(c, p, in_mode, epi, prepare);
  } else {
    if (ny == 1) return dispatch_epi<kWQ4, 1, 2, 8>(c, p, in_mode, epi, prepare);
    if (ny == 2) return dispatch_epi<kWQ4, 2, 2, 8>(c, p, in_mode, epi, prepare);
    if (ny == 4) return dispatch_epi<kWQ4, 4, 1, 16>(c, p, in_mode, epi, prepare);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int gemm_tc_ny(int wfmt, int batch) {
  const int ny = (batch + 7) / 8;
  if (wfmt == kWBf16) return ny <= 2 ? ny : 0;
  return ny <= 1 ? 1 : ny <= 2 ? 2 : ny <= 4 ? 4 : 0;
}

int gemm_tc_rows_per_block(int wfmt, int) { return wfmt == kWQ4 ? 256 : 128; }

int gemm_tc_block_tokens(int wfmt) { return wfmt == kWQ4 ? 32 : 16; }

int gemm_tc_chunk(int ny) { return ny == 1 ? 1024 : 512; }

cudaError_t launch_gemm_tc(const LaunchCtx& c, const GemmParams& p, int wfmt, int in_mode, int epi) {
  return dispatch(c, p, wfmt, in_mode, epi, false);
}

cudaError_t prepare_gemm_tc(const GemmParams& p, int wfmt, int in_mode, int epi) {
  return dispatch(LaunchCtx{nullptr, false}, p, wfmt, in_mode, epi, true);
}

}  // namespace dec

// Step prologue (embedding gather, RoPE table, status checks), create-time weight
// packing, the dequant test hook and the greedy feedback helper.
#include "dec_internal.cuh"
#include "q4.cuh"

namespace dec {

// ---------------------------------------------------------------- embedding gather
// Butter architecture.md, "SINGLE-TOKEN DECODE": h = embed_tokens[prev_token].
// Also: per-8-row sums of squares of h (consumed by the first layer's fused
// RMSNorm), the (cos, sin) table of this step's RoPE angles pos * theta^(-2i/d)
// evaluated in double precision, reset of the argmax key, and range checks.
__global__ void __launch_bounds__(256) k_embed(EmbedParams p) {
  tl_mark(p.tl, 0);
  griddep_wait();  // first kernel of a step: nothing upstream inside the graph
  tl_mark(p.tl, 1);
  const int b = blockIdx.x;
  const int T = p.T > 1 ? p.T : 1;
  int tok = p.tokens[b];
  int pos = p.positions[b / T] + b % T;
  if (tok < 0 || tok >= p.V) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadToken);
    tok = tok < 0 ? 0 : p.V - 1;
  }
  if (pos < 0 || pos >= p.max_ctx) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadPos);
    pos = pos < 0 ? 0 : p.max_ctx - 1;
  }
  const __nv_bfloat16* row = p.embed + static_cast<size_t>(tok) * p.H;
  float* hb = p.h + static_cast<size_t>(b) * p.H;
  const int ngroups = p.H / kResGroup;
  for (int gidx = threadIdx.x; gidx < ngroups; gidx += blockDim.x) {
    uint4 u = *reinterpret_cast<const uint4*>(row + gidx * kResGroup);
    float v[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y),
                  bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)};
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
    float4* dst = reinterpret_cast<float4*>(hb + gidx * kResGroup);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    p.sumsq[static_cast<size_t>(b) * ngroups + gidx] = ss;
    if (p.xhl_out) {  // batched path: the first projection's input h * in_norm as hi + lo planes
      const size_t plane = static_cast<size_t>(gridDim.x) * p.H;
      __nv_bfloat16* hi = p.xhl_out + static_cast<size_t>(b) * p.H + gidx * kResGroup;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float u = v[i] * __bfloat162float(p.norm_w0[gidx * kResGroup + i]);
        const __nv_bfloat16 uh = __float2bfloat16_rn(u);
        hi[i] = uh;
        hi[plane + i] = __float2bfloat16_rn(u - __bfloat162float(uh));
      }
    }
  }
  for (int i = threadIdx.x; i < p.half_d; i += blockDim.x) {
    double ang = static_cast<double>(pos) * p.inv_freq[i];
    double s, c;
    sincos(ang, &s, &c);
    p.rope[static_cast<size_t>(b) * p.half_d + i] = make_float2(static_cast<float>(c), static_cast<float>(s));
  }
  if (threadIdx.x == 0) p.amax_key[b] = 0ull;
  griddep_launch_dependents();
  tl_mark(p.tl, 2);
}

cudaError_t launch_embed(const LaunchCtx& c, const EmbedParams& p, int B) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_embed, p);
}

// ---------------------------------------------------------------- RoPE table (stand-alone attention entry points)
__global__ void k_rope_table(const int32_t* positions, int half_d, int max_ctx, double theta, float2* rope,
                             unsigned* status) {
  const int b = blockIdx.x;
  int pos = positions[b];
  if (pos < 0 || pos >= max_ctx) {
    if (threadIdx.x == 0 && status) atomicOr(status, kStatusBadPos);
    pos = pos < 0 ? 0 : max_ctx - 1;
  }
  for (int i = threadIdx.x; i < half_d; i += blockDim.x) {
    const double inv = pow(theta, -2.0 * i / (2.0 * half_d));
    double s, c;
    sincos(static_cast<double>(pos) * inv, &s, &c);
    rope[static_cast<size_t>(b) * half_d + i] = make_float2(static_cast<float>(c), static_cast<float>(s));
  }
}

cudaError_t launch_rope_table(cudaStream_t s, const int32_t* positions, int batch, int head_dim, int max_ctx,
                              float theta, float2* rope, unsigned* status) {
  k_rope_table<<<batch, 64, 0, s>>>(positions, head_dim / 2, max_ctx, static_cast<double>(theta), rope, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- packing (create time)
// Row p of the packed matrix takes, with interleave block IB > 0,
//   block = p / (2 IB), w = p % (2 IB): w < IB ? A[block IB + w] : B[block IB + w - IB]
// and with IB == 0 simply A[p].
__device__ __forceinline__ void packed_source(int p, int ib, int& which, int& src_row) {
  if (ib == 0) {
    which = 0;
    src_row = p;
  } else {
    int block = p / (2 * ib), w = p % (2 * ib);
    which = w < ib ? 0 : 1;
    src_row = block * ib + (w < ib ? w : w - ib);
  }
}

__global__ void k_pack_rows_bf16(__nv_bfloat16* dst, const __nv_bfloat16* a, const __nv_bfloat16* b,
                                 int rows_out, int K, int ib) {
  const int p = blockIdx.x;
  if (p >= rows_out) return;
  int which, r;
  packed_source(p, ib, which, r);
  const uint4* src = reinterpret_cast<const uint4*>((which ? b : a) + static_cast<size_t>(r) * K);
  uint4* d = reinterpret_cast<uint4*>(dst + static_cast<size_t>(p) * K);
  for (int i = threadIdx.x; i < K / 8; i += blockDim.x) d[i] = src[i];
}

cudaError_t pack_rows_bf16(cudaStream_t s, __nv_bfloat16* dst, const __nv_bfloat16* src_a,
                           const __nv_bfloat16* src_b, int rows_out, int K, int interleave_block) {
  if (rows_out == 0) return cudaSuccess;
  k_pack_rows_bf16<<<rows_out, 128, 0, s>>>(dst, src_a, src_b, rows_out, K, interleave_block);
  return cudaGetLastError();
}

__global__ void k_pack_rows_q4(uint32_t* dst_w, uint32_t* dst_sb, const uint32_t* wa, const __nv_bfloat16* sa,
                               const __nv_bfloat16* ba, const uint32_t* wb, const __nv_bfloat16* sbb,
                               const __nv_bfloat16* bb, int rows_out, int K, int ib) {
  const int p = blockIdx.x;
  if (p >= rows_out) return;
  int which, r;
  packed_source(p, ib, which, r);
  const uint32_t* w = which ? wb : wa;
  const __nv_bfloat16* sc = which ? sbb : sa;
  const __nv_bfloat16* bi = which ? bb : ba;
  const int nw = K / 8, ng = K / kGroup;
  const uint4* src = reinterpret_cast<const uint4*>(w + static_cast<size_t>(r) * nw);
  uint4* d = reinterpret_cast<uint4*>(dst_w + static_cast<size_t>(p) * nw);
  for (int i = threadIdx.x; i < nw / 4; i += blockDim.x) d[i] = src[i];
  for (int g = threadIdx.x; g < ng; g += blockDim.x) {
    uint32_t s16 = __bfloat16_as_ushort(sc[static_cast<size_t>(r) * ng + g]);
    uint32_t b16 = __bfloat16_as_ushort(bi[static_cast<size_t>(r) * ng + g]);
    dst_sb[static_cast<size_t>(p) * ng + g] = s16 | (b16 << 16);
  }
}

cudaError_t pack_rows_q4(cudaStream_t s, uint32_t* dst_w, uint32_t* dst_sb, const uint32_t* src_w_a,
                         const __nv_bfloat16* sc_a, const __nv_bfloat16* bi_a, const uint32_t* src_w_b,
                         const __nv_bfloat16* sc_b, const __nv_bfloat16* bi_b, int rows_out, int K,
                         int interleave_block) {
  if (rows_out == 0) return cudaSuccess;
  k_pack_rows_q4<<<rows_out, 128, 0, s>>>(dst_w, dst_sb, src_w_a, sc_a, bi_a, src_w_b, sc_b, bi_b, rows_out, K,
                                          interleave_block);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- dequant test hook
// out[r][k] (canonical row r of one linear) from the packed copy, with the GEMV's
// code extraction and a single rounding: fmaf(scale, q, bias).
__global__ void k_debug_dequant(float* out, const void* w, const uint32_t* sb, int wfmt, int rows_out, int K,
                                int row_offset, int ib, int which_half) {
  const int r = blockIdx.x;
  if (r >= rows_out) return;
  int p;
  if (which_half < 0) {
    p = row_offset + r;
  } else {
    int block = r / ib, within = r % ib;
    p = row_offset + block * 2 * ib + which_half * ib + within;
  }
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    float v;
    if (wfmt == kWBf16) {
      const __nv_bfloat16* wb = static_cast<const __nv_bfloat16*>(w);
      v = __bfloat162float(wb[static_cast<size_t>(p) * K + k]);
    } else {
      const uint32_t* ww = static_cast<const uint32_t*>(w);
      uint32_t word = ww[static_cast<size_t>(p) * (K / 8) + k / 8];
      float q = q4_code_plus128_rt(word, k % 8) - 128.0f;
      uint32_t g = sb[static_cast<size_t>(p) * (K / kGroup) + k / kGroup];
      v = fmaf(sb_scale(g), q, sb_bias(g));
    }
    out[static_cast<size_t>(r) * K + k] = v;
  }
}

cudaError_t debug_dequant(cudaStream_t s, float* out, const void* w, const uint32_t* sb, int wfmt, int rows_out,
                          int K, int row_offset, int interleave_block, int which_half) {
  k_debug_dequant<<<rows_out, 256, 0, s>>>(out, w, sb, wfmt, rows_out, K, row_offset, interleave_block,
                                           which_half);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- fragment packing (batched path)
// bf16: tile (16 rows x 16 inputs) = 32 lanes x 4 registers; lane (g, t) register r holds
// rows g + 8 (r & 1), inputs 2t + 8 (r >> 1) and the next input, first in the low half.
__global__ void k_pack_frag_bf16(uint32_t* dst, const __nv_bfloat16* a, const __nv_bfloat16* b, int rows_out,
                                 int npad, int K, int ib, int row_off) {
  const int kt_n = K / 16;
  const size_t total = static_cast<size_t>(npad / 16) * kt_n * 128;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int reg = static_cast<int>(idx & 3), lane = static_cast<int>((idx >> 2) & 31);
    const size_t tile = idx >> 7;
    const int kt = static_cast<int>(tile % kt_n), rtl = static_cast<int>(tile / kt_n);
    const int g = lane >> 2, t = lane & 3;
    const int row = 16 * rtl + g + 8 * (reg & 1), col = 16 * kt + 2 * t + 8 * (reg >> 1);
    uint32_t v = 0;
    if (row < rows_out) {
      int which, r;
      packed_source(row, ib, which, r);
      const __nv_bfloat16* src = (which ? b : a) + static_cast<size_t>(r) * K + col;
      v = static_cast<uint32_t>(__bfloat16_as_ushort(src[0])) |
          (static_cast<uint32_t>(__bfloat16_as_ushort(src[1])) << 16);
    }
    dst[((static_cast<size_t>(row_off / 16 + rtl) * kt_n + kt) * 32 + lane) * 4 + reg] = v;
  }
}

cudaError_t pack_frag_bf16(cudaStream_t s, uint32_t* dst, const __nv_bfloat16* src_a, const __nv_bfloat16* src_b,
                           int rows_out, int npad, int K, int interleave_block, int dst_row_offset, int) {
  k_pack_frag_bf16<<<1024, 256, 0, s>>>(dst, src_a, src_b, rows_out, npad, K, interleave_block, dst_row_offset);
  return cudaGetLastError();
}

// 4-bit: tile (16 rows x 64 inputs) = 512 bytes of codes + 64 bytes of (scale, bias).
// Lane (g, t), k-step j: one word whose bits 4i..4i+3 and 16+4i..16+4i+3 hold A register i:
// i = 0: row g, inputs c, c+1; i = 1: row g+8, inputs c, c+1; i = 2: row g, inputs c+8, c+9;
// i = 3: row g+8, inputs c+8, c+9 (c = 16 j + 2 t within the group).  Then for each g the
// bf16 scale and bias of row g followed by those of row g+8.
__global__ void k_pack_frag_q4(unsigned char* dst, const uint32_t* wa, const __nv_bfloat16* sa,
                               const __nv_bfloat16* ba, const uint32_t* wb, const __nv_bfloat16* sbb,
                               const __nv_bfloat16* bb, int rows_out, int npad, int K, int ib, int row_off) {
  const int gk_n = K / kGroup;
  const size_t total = static_cast<size_t>(npad / 16) * gk_n * 32;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int lane = static_cast<int>(idx & 31);
    const size_t tile = idx >> 5;
    const int gk = static_cast<int>(tile % gk_n), rtl = static_cast<int>(tile / gk_n);
    const int g = lane >> 2, t = lane & 3;
    const int r0 = 16 * rtl + g, r1 = r0 + 8;
    auto code = [&](int row, int col) -> uint32_t {
      if (row >= rows_out) return 0u;
      int which, r;
      packed_source(row, ib, which, r);
      const uint32_t w = (which ? wb : wa)[static_cast<size_t>(r) * (K / 8) + col / 8];
      return (w >> (4 * (col % 8))) & 0xfu;
    };
    unsigned char* tp = dst + (static_cast<size_t>(row_off / 16 + rtl) * gk_n + gk) * 576;
    for (int j = 0; j < 4; ++j) {
      const int c = gk * kGroup + 16 * j + 2 * t;
      const uint32_t word = code(r0, c) | (code(r0, c + 1) << 16) | (code(r1, c) << 4) | (code(r1, c + 1) << 20) |
                            (code(r0, c + 8) << 8) | (code(r0, c + 9) << 24) | (code(r1, c + 8) << 12) |
                            (code(r1, c + 9) << 28);
      reinterpret_cast<uint32_t*>(tp + lane * 16)[j] = word;
    }
    if (t == 0) {
      auto sbpair = [&](int row) -> uint32_t {
        if (row >= rows_out) return 0u;
        int which, r;
        packed_source(row, ib, which, r);
        const size_t o = static_cast<size_t>(r) * gk_n + gk;
        return static_cast<uint32_t>(__bfloat16_as_ushort((which ? sbb : sa)[o])) |
               (static_cast<uint32_t>(__bfloat16_as_ushort((which ? bb : ba)[o])) << 16);
      };
      uint2 v;
      v.x = sbpair(r0);
      v.y = sbpair(r1);
      *reinterpret_cast<uint2*>(tp + 512 + g * 8) = v;
    }
  }
}

cudaError_t pack_frag_q4(cudaStream_t s, unsigned char* dst, const uint32_t* w_a, const __nv_bfloat16* sc_a,
                         const __nv_bfloat16* bi_a, const uint32_t* w_b, const __nv_bfloat16* sc_b,
                         const __nv_bfloat16* bi_b, int rows_out, int K, int interleave_block, int dst_row_offset,
                         int npad) {
  k_pack_frag_q4<<<1024, 256, 0, s>>>(dst, w_a, sc_a, bi_a, w_b, sc_b, bi_b, rows_out, npad, K, interleave_block,
                                      dst_row_offset);
  return cudaGetLastError();
}

// dequant test hook for the fragment layouts: canonical row r, input k
__global__ void k_debug_dequant_frag(float* out, const void* w, int wfmt, int rows_out, int K, int row_offset, int ib,
                                     int which_half) {
  const int r = blockIdx.x;
  if (r >= rows_out) return;
  int p;
  if (which_half < 0) {
    p = row_offset + r;
  } else {
    const int block = r / ib, within = r % ib;
    p = row_offset + block * 2 * ib + which_half * ib + within;
  }
  const int rt = p / 16, gg = (p % 16) % 8, hi = (p % 16) / 8;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    float v;
    if (wfmt == kWBf16) {
      const int kt = k / 16, kk = k % 16;
      const int lane = 4 * gg + (kk % 8) / 2, reg = hi + 2 * (kk / 8);
      const uint32_t u =
          static_cast<const uint32_t*>(w)[((static_cast<size_t>(rt) * (K / 16) + kt) * 32 + lane) * 4 + reg];
      v = (kk & 1) ? bf16_hi(u) : bf16_lo(u);
    } else {
      const int gk = k / kGroup, kq = k % kGroup, j = kq / 16, kk = kq % 16;
      const int lane = 4 * gg + (kk % 8) / 2;
      const unsigned char* tp = static_cast<const unsigned char*>(w) + (static_cast<size_t>(rt) * (K / kGroup) + gk) * 576;
      const uint32_t word = reinterpret_cast<const uint32_t*>(tp + lane * 16)[j];
      const uint32_t q2 = q4_pair_bf16(word, 4 * (hi + 2 * (kk / 8)));
      const float q = (kk & 1) ? bf16_hi(q2) : bf16_lo(q2);
      const uint2 sbv = *reinterpret_cast<const uint2*>(tp + 512 + gg * 8);
      const uint32_t sbw = hi ? sbv.y : sbv.x;
      v = fmaf(sb_scale(sbw), q, sb_bias(sbw));
    }
    out[static_cast<size_t>(r) * K + k] = v;
  }
}

cudaError_t debug_dequant_frag(cudaStream_t s, float* out, const void* w, int wfmt, int rows_out, int K,
                               int row_offset, int interleave_block, int which_half) {
  k_debug_dequant_frag<<<rows_out, 256, 0, s>>>(out, w, wfmt, rows_out, K, row_offset, interleave_block, which_half);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- greedy feedback
__global__ void k_advance(const int32_t* argmax, int32_t* tokens, int32_t* positions, int batch) {
  int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) {
    tokens[b] = argmax[b];
    positions[b] += 1;
  }
}

// Profiling aid: one thread sleeps until `ns` nanoseconds of %globaltimer have passed
// (at most 2 ns / 256 sleeps of 256 ns), so that a stream held on it fills up with the
// host's launches before the first of them runs.
__global__ void k_hold(unsigned long long ns) {
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  const unsigned long long max_iter = ns / 128 + 1;
  for (unsigned long long i = 0; i < max_iter; ++i) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 >= ns) break;
    __nanosleep(256);
  }
}

cudaError_t launch_hold(cudaStream_t s, unsigned long long ns) {
  k_hold<<<1, 1, 0, s>>>(ns);
  return cudaGetLastError();
}

// A bounded wait that can only run out: one thread initialises an mbarrier that nothing ever
// arrives on and polls its first phase `polls` times, then sets the time-out bit of the status
// word, as every bounded wait of the tensor-memory kernels does when a copy or an MMA never
// completes.  The host reads it through dec_get_device_status (DEC_ERR_TIMEOUT); the context
// stays usable.
__global__ void k_force_timeout(unsigned* status, int polls) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(1) : "memory");
  bool done = false;
  for (int i = 0; i < polls && !done; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(b), "r"(0u)
        : "memory");
    done = ok != 0;
  }
  if (!done) atomicOr(status, kStatusTimeout);
}

cudaError_t launch_force_timeout(cudaStream_t s, unsigned* status, int polls) {
  k_force_timeout<<<1, 1, 0, s>>>(status, polls);
  return cudaGetLastError();
}

cudaError_t launch_advance(cudaStream_t s, const int32_t* argmax, int32_t* tokens, int32_t* positions,
                           int batch) {
  k_advance<<<(batch + 127) / 128, 128, 0, s>>>(argmax, tokens, positions, batch);
  return cudaGetLastError();
}

}  // namespace dec

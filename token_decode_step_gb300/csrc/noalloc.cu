// dec_attention_noalloc: the stand-alone fused attention (as dec_attention) for
// callers that cannot allocate device memory.  Its scratch -- the RoPE (cos, sin)
// table that the first of its two kernels writes and the attention kernel reads
// -- lives in one file-scope device array instead of a caller workspace.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "dec_internal.cuh"

using namespace dec;

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB: RoPE tables of up to 2048 sequences (head_dim 128)
constexpr int kMaxDevices = 64;

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
unsigned char* g_scratch_addr[kMaxDevices];  // device address of g_attn_scratch, per device; null until set up

// Per-device set-up with that device current: the device address of the array
// (in host code the name g_attn_scratch is only a host-side stand-in) and the
// attention kernels' shared-memory limit.
dec_status setup_device(int dev, unsigned char** addr) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess || !p) {
      set_last_error("dec_attention_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      return DEC_ERR_CUDA;
    }
    const int dims[2] = {64, 128};
    const int groups[3] = {1, 2, 4};
    const int fmts[2] = {DEC_KV_BF16, DEC_KV_AFFINE8_G64};
    for (int f : fmts)
      for (int d : dims)
        for (int g : groups)
          if ((e = prepare_attention(d, g, f)) != cudaSuccess) {
            set_last_error("dec_attention_noalloc: kernel set-up failed: %s", cudaGetErrorString(e));
            return DEC_ERR_CUDA;
          }
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
  }
  *addr = g_scratch_addr[dev];
  return DEC_OK;
}

}  // namespace

extern "C" dec_status dec_attention_noalloc(const dec_config* cfg, int layer, const float* qkv, const void* q_norm,
                                            const void* k_norm, const int32_t* positions, void* kv_cache, float* out,
                                            dec_stream_t stream) {
  // the same config checks as dec_attention (tokens_per_seq > 1 included)
  dec_status vst = validate_attention_cfg(cfg, layer);
  if (vst != DEC_OK) return vst;
  const dec_config& c = *cfg;
  if (!qkv || !q_norm || !k_norm || !positions || !kv_cache || !out ||
      (reinterpret_cast<uintptr_t>(kv_cache) & 15u)) {
    set_last_error("dec_attention_noalloc: NULL pointer or kv_cache not 16-byte aligned");
    return DEC_ERR_INVALID_ARG;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_error("dec_attention_noalloc: cannot query the current device: %s", cudaGetErrorString(e));
    return DEC_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_last_error("dec_attention_noalloc: device ordinal %d above %d", dev, kMaxDevices - 1);
    return DEC_ERR_UNSUPPORTED;
  }

  // scratch: the RoPE table, batch x head_dim/2 x (cos, sin)
  const size_t total = static_cast<size_t>(c.batch) * (c.head_dim / 2) * 8;
  if (total > kNoAllocScratchBytes) {
    set_last_error("dec_attention_noalloc: batch %d needs %zu bytes of scratch, above the fixed %zu-byte array "
                   "(use dec_attention with a workspace)",
                   c.batch, total, kNoAllocScratchBytes);
    return DEC_ERR_UNSUPPORTED;
  }

  unsigned char* scratch = nullptr;
  dec_status st = setup_device(dev, &scratch);
  if (st != DEC_OK) return st;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  float2* rope = reinterpret_cast<float2*>(scratch);  // fully rewritten by every call
  if ((e = launch_rope_table(cs, positions, c.batch, c.head_dim, c.max_ctx, c.rope_theta, rope, nullptr)) !=
      cudaSuccess) {
    set_last_error("dec_attention_noalloc: RoPE table launch failed: %s", cudaGetErrorString(e));
    return DEC_ERR_CUDA;
  }
  AttnParams ap{};
  ap.qkv = qkv;
  ap.q_norm = static_cast<const __nv_bfloat16*>(q_norm);
  ap.k_norm = static_cast<const __nv_bfloat16*>(k_norm);
  ap.rope = rope;
  ap.positions = positions;
  attn_set_cache(ap, c, kv_cache);
  ap.layer = layer;
  ap.B = c.batch;
  ap.nq = c.n_q_heads;
  ap.nkv = c.n_kv_heads;
  ap.max_ctx = c.max_ctx;
  ap.eps = c.rms_eps;
  ap.out = out;
  ap.status = nullptr;
  if ((e = launch_attention(LaunchCtx{cs, false}, ap, c.head_dim)) != cudaSuccess) {
    set_last_error("dec_attention_noalloc: attention launch failed: %s", cudaGetErrorString(e));
    return DEC_ERR_CUDA;
  }
  return DEC_OK;
}

// C ABI of the decode step: handle lifetime, argument checks, weight packing,
// the per-step launch sequence, CUDA-graph capture/replay and profiling.
//
// The launch sequence follows Butter architecture.md, figure "SINGLE-TOKEN
// DECODE" (gather -> per layer: rms_norm+qkv, rope+append+sdpa, o+add,
// rms_norm+gate/up+silu_mul, down+add -> rms_norm+lm_head -> argmax), with the
// norms and elementwise steps fused into the neighbouring kernels.  The page's
// "one command buffer per token" becomes one CUDA graph per step, and the
// argument-buffer idea (weights bound once, per-token state small) becomes a
// graph whose kernel parameters are fixed per pointer set.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "dec_internal.cuh"

using namespace dec;

// ---------------------------------------------------------------- errors

static thread_local char g_err[512] = "";

static void set_err(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

namespace dec {
void set_last_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}
// Checks of a config for the stand-alone attention entry points (dec_attention and
// dec_attention_noalloc share them, so that the two cannot drift apart).
dec_status validate_attention_cfg(const dec_config* c, int layer) {
  if (!c) {
    set_last_error("config is NULL");
    return DEC_ERR_INVALID_ARG;
  }
  if (c->n_layers < 1 || c->batch < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1 || c->max_ctx < 1 ||
      layer < 0 || layer >= c->n_layers || !(c->rms_eps > 0.f) || !(c->rope_theta > 1.f)) {
    set_last_error("attention: sizes must be positive, 0 <= layer < n_layers, rms_eps > 0, rope_theta > 1");
    return DEC_ERR_INVALID_ARG;
  }
  if (c->n_q_heads % c->n_kv_heads != 0) {
    set_last_error("n_q_heads (%d) must be a multiple of n_kv_heads (%d)", c->n_q_heads, c->n_kv_heads);
    return DEC_ERR_INVALID_ARG;
  }
  if (c->tokens_per_seq > 1) {
    set_last_error("attention: the stand-alone entry points take tokens_per_seq 0 or 1");
    return DEC_ERR_UNSUPPORTED;
  }
  if (c->kv_fmt != DEC_KV_BF16 && c->kv_fmt != DEC_KV_AFFINE8_G64) {
    set_last_error("attention: unknown kv_fmt %d", c->kv_fmt);
    return DEC_ERR_INVALID_ARG;
  }
  if (c->kv_fmt == DEC_KV_AFFINE8_G64 && c->max_ctx % 16 != 0) {
    set_last_error("attention: the affine 8-bit KV cache needs max_ctx to be a multiple of 16 (got %d)", c->max_ctx);
    return DEC_ERR_UNSUPPORTED;
  }
  const int G = c->n_q_heads / c->n_kv_heads;
  if ((G != 1 && G != 2 && G != 4) || (c->head_dim != 64 && c->head_dim != 128)) {
    set_last_error("attention: head_dim must be 64 or 128 and n_q_heads/n_kv_heads 1, 2 or 4");
    return DEC_ERR_UNSUPPORTED;
  }
  return DEC_OK;
}

}  // namespace dec

#define DEC_CUDA(call)                                                                     \
  do {                                                                                     \
    cudaError_t e_ = (call);                                                               \
    if (e_ != cudaSuccess) {                                                               \
      set_err("%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
      return DEC_ERR_CUDA;                                                                 \
    }                                                                                      \
  } while (0)

// ---------------------------------------------------------------- handle

namespace {

struct PackedLinear {
  alignas(64) unsigned char tmap[128] = {};  // tcgen05 path: TMA tensor map of w (bf16 [N][K])
  int tile_n = 128;                            // tcgen05 path: weight rows per tile (the map's box)
  void* w = nullptr;       // batch 1 and tcgen05 path: bf16 [N][K] or uint32 [N][K/8]; batched: fragment tiles
  uint32_t* sb = nullptr;  // batch-1 q4 only: [N][K/64]
  int N = 0, K = 0, S = 1;
  int Npad = 0, KC = 0;    // batched path: rows padded to 16, inputs staged per chunk
  size_t w_bytes = 0, sb_bytes = 0;  // sizes of the two regions (sb_bytes 0 when sb is null)
  bool frag = false;       // fragment tiles of the mma.sync batched kernel (else row-major)
  bool q4tc = false;       // launched on the tcgen05 4-bit kernel (k_gemm_q4tc)
};

struct PackedLayer {
  __nv_bfloat16 *in_norm, *post_norm, *q_norm, *k_norm;
  PackedLinear qkv, o, gateup, down;
};

struct StepPtrs {
  const int32_t* tokens;
  const int32_t* positions;
  void* kv;
  float* logits;
  int32_t* argmax;
  bool operator==(const StepPtrs& o) const {
    return tokens == o.tokens && positions == o.positions && kv == o.kv && logits == o.logits &&
           argmax == o.argmax;
  }
};

struct Launch {
  int cls;
};

}  // namespace

struct dec_handle {
  dec_config cfg{};
  int device = 0;
  int num_sms = 0;
  int wfmt = 0;
  int tps = 1;   // tokens per sequence (1: decode; 2..8: verify)
  int rows = 1;  // batch * tps: rows of every projection
  int tblocks = 1;  // batched path: token blocks per projection launch
  // tcgen05 path (bf16 weights, at least a 128-token tile of rows): row-major weights and
  // TMA tensor maps of the three activation hi/lo planes (inputs of QKV / gate_up / lm_head,
  // of O, of down)
  bool umma = false;
  // batched decode (2..32 rows) with 4-bit weights on models of hidden >= 2048: some or all
  // projections on tcgen05 over expanded code tiles (PackedLinear::q4tc); their weights stay in
  // the batch-1 row-major packing, read by TMA (the codes) and plain loads (scale and bias); the
  // activation maps (map_u, map_o, map_g) have 32-row boxes
  bool q4tc = false;
  // the same for bf16 weights at 1..32 rows (k_gemm_btc): row-major weights read by TMA
  bool btc = false;
  alignas(64) unsigned char map_u[128] = {}, map_o[128] = {}, map_g[128] = {};
  // batch 1: the QKV GEMV prefetches the attention's cached K/V rows into L2 (when a
  // layer's K/V at max_ctx takes at most a quarter of L2)
  bool kv_prefetch = false;
  // prefill chunks (16+ tokens per sequence, bf16 cache): the causal attention that stages
  // each K/V tile once for 64 query rows (k_attn_prefill) instead of one decode attention
  // per row
  bool attn_prefill = false;

  // packed weights (one allocation)
  unsigned char* wmem = nullptr;
  size_t wbytes = 0;
  __nv_bfloat16* embed = nullptr;
  __nv_bfloat16* final_norm = nullptr;
  PackedLinear lm_head;
  std::vector<PackedLayer> layers;
  // workspace (one allocation)
  unsigned char* ws = nullptr;
  float* h = nullptr;
  float* qkv = nullptr;
  float* attn_o = nullptr;
  float* g = nullptr;
  float* sumsq = nullptr;
  // batched path: next-consumer inputs as bf16 hi, lo planes
  __nv_bfloat16* xh_u = nullptr;  // [2][B][H]: h times the next norm weight
  __nv_bfloat16* xh_o = nullptr;  // [2][B][nq d]: attention output
  __nv_bfloat16* xh_g = nullptr;  // [2][B][I]: SwiGLU output
  float* gemv_partials = nullptr;
  unsigned* gemv_counters = nullptr;
  float2* rope = nullptr;
  double* inv_freq = nullptr;
  unsigned long long* amax_key = nullptr;
  unsigned* status = nullptr;
  // graph state
  bool graph_mode = true;
  cudaStream_t cap_stream = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  bool have_graph = false;
  StepPtrs captured{};
  // dec_step_host: staging int32 [rows tokens | batch positions | rows argmax], pinned on
  // the host and on the device (allocated by the first call), and the graph that copies
  // in, runs the step and copies the argmax back
  int32_t* io_host = nullptr;
  int32_t* io_dev = nullptr;
  cudaGraph_t hgraph = nullptr;
  cudaGraphExec_t hexec = nullptr;
  bool have_hgraph = false;
  StepPtrs hcaptured{};
  // profiling: events around every launch; the stream is held (by a sleeping kernel
  // on hold_stream) until the host has enqueued the whole step
  std::vector<cudaEvent_t> events;
  cudaStream_t hold_stream = nullptr;
  cudaEvent_t hold_ev = nullptr;
  // debug: stop an eager step after this many launches (-1: no limit)
  int launch_limit = -1;
  // debug: per-launch %globaltimer stamps (device, 3 per launch) or null
  unsigned long long* timeline = nullptr;
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

double wbytes_per_elem(int fmt) { return fmt == DEC_W_BF16 ? 2.0 : 0.5 + 4.0 / kGroup; }

size_t linear_bytes_tc(int fmt, int N, int K) {
  const size_t npad = (static_cast<size_t>(N) + 15) / 16 * 16;
  if (fmt == DEC_W_BF16) return align_up(npad * K * 2, 256);
  return align_up(npad / 16 * (K / kGroup) * 576, 256);
}

size_t linear_bytes(int fmt, int N, int K) {
  if (fmt == DEC_W_BF16) return align_up(static_cast<size_t>(N) * K * 2, 256);
  return align_up(static_cast<size_t>(N) * K / 2, 256) + align_up(static_cast<size_t>(N) * (K / kGroup) * 4, 256);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dec_status validate(const dec_config* c) {
  if (!c) {
    set_err("config is NULL");
    return DEC_ERR_INVALID_ARG;
  }
  if (c->n_layers < 1 || c->hidden < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 1 ||
      c->intermediate < 1 || c->vocab < 1 || c->batch < 1 || c->max_ctx < 1) {
    set_err("config sizes must be positive");
    return DEC_ERR_INVALID_ARG;
  }
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 1.f) || !std::isfinite(c->rms_eps) || !std::isfinite(c->rope_theta)) {
    set_err("rms_eps must be > 0 and rope_theta > 1");
    return DEC_ERR_INVALID_ARG;
  }
  if (c->linear_fmt != DEC_W_BF16 && c->linear_fmt != DEC_W_AFFINE4_G64) {
    set_err("unknown linear_fmt %d", c->linear_fmt);
    return DEC_ERR_INVALID_ARG;
  }
  if (c->proj_kernels < DEC_PROJ_AUTO || c->proj_kernels > DEC_PROJ_TCGEN05) {
    set_err("unknown proj_kernels %d", c->proj_kernels);
    return DEC_ERR_INVALID_ARG;
  }
  if (c->n_q_heads % c->n_kv_heads != 0) {
    set_err("n_q_heads (%d) must be a multiple of n_kv_heads (%d)", c->n_q_heads, c->n_kv_heads);
    return DEC_ERR_INVALID_ARG;
  }
  const int G = c->n_q_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4) {
    set_err("query heads per KV head must be 1, 2 or 4 (got %d)", G);
    return DEC_ERR_UNSUPPORTED;
  }
  if (c->head_dim != 64 && c->head_dim != 128) {
    set_err("head_dim must be 64 or 128 (got %d)", c->head_dim);
    return DEC_ERR_UNSUPPORTED;
  }
  if (c->hidden % 64 || c->intermediate % 64) {
    set_err("hidden and intermediate must be multiples of 64");
    return DEC_ERR_UNSUPPORTED;
  }
  if (c->kv_fmt != DEC_KV_BF16 && c->kv_fmt != DEC_KV_AFFINE8_G64) {
    set_err("unknown kv_fmt %d", c->kv_fmt);
    return DEC_ERR_INVALID_ARG;
  }
  if (c->kv_fmt == DEC_KV_AFFINE8_G64 && c->max_ctx % 16 != 0) {
    set_err("the affine 8-bit KV cache needs max_ctx to be a multiple of 16 (got %d)", c->max_ctx);
    return DEC_ERR_UNSUPPORTED;
  }
  if (c->tokens_per_seq < 0 || c->tokens_per_seq > kMaxTokensPerSeq) {
    set_err("tokens_per_seq must be 0..%d (got %d)", kMaxTokensPerSeq, c->tokens_per_seq);
    return c->tokens_per_seq < 0 ? DEC_ERR_INVALID_ARG : DEC_ERR_UNSUPPORTED;
  }
  const long long rows = static_cast<long long>(c->batch) * (c->tokens_per_seq > 1 ? c->tokens_per_seq : 1);
  if (rows > kMaxRows) {
    set_err("batch %d x tokens_per_seq %d = %lld rows, at most %d per step", c->batch, c->tokens_per_seq, rows,
            kMaxRows);
    return DEC_ERR_UNSUPPORTED;
  }
  if (static_cast<long long>(c->max_ctx) * c->n_kv_heads * c->batch * c->head_dim > (1ll << 40)) {
    set_err("KV cache too large");
    return DEC_ERR_UNSUPPORTED;
  }
  return DEC_OK;
}

dec_status check_linear(const dec_linear& l, int fmt, const char* name, int layer) {
  if (!l.w || !aligned16(l.w)) {
    set_err("layer %d %s: weight pointer NULL or not 16-byte aligned", layer, name);
    return DEC_ERR_INVALID_ARG;
  }
  if (fmt == DEC_W_AFFINE4_G64 && (!l.scales || !l.biases)) {
    set_err("layer %d %s: affine 4-bit linear needs scales and biases", layer, name);
    return DEC_ERR_INVALID_ARG;
  }
  return DEC_OK;
}

// K splits of a batch-1 GEMV: split only while the CTAs would cover fewer than half the
// SMs.  Every split costs a round trip through the partial sums (fence, ticket, reload:
// about 2 us measured on the 1024-row projections, more than the idle SMs give back).
// Which projections of a step with `rows` rows run on the tcgen05 decode kernels.  2..32 rows (a
// batch of sequences, or the rows of a verify step) at hidden >= 2048: tcgen05 on the batched
// path's hi/lo activation planes, 4-bit codes expanded into tensor memory (k_gemm_q4tc) or bf16
// weights streamed by TMA (k_gemm_btc).  DEC_PROJ_TCGEN05 puts every projection there.
// DEC_PROJ_AUTO takes what measured faster side by side on one GPU: with 4-bit weights from 16
// rows on (measured at 32), the gate/up and lm_head projections on tcgen05 and the others on
// mma.sync (8B, 32 rows: gate/up 69 against 84 us, lm_head 0.30 against 0.40 ms; q/k/v, o and
// down 37-53 against 35-49 us), with bf16 weights every projection on mma.sync (8 rows: 3.79
// against 5.20 ms a step).  One row stays on the batch-1 GEMV.
struct ProjPlan {
  bool q4tc_all = false;  // every projection on k_gemm_q4tc
  bool q4tc_gu = false;   // the gate/up and lm_head projections on k_gemm_q4tc
  bool btc = false;       // every projection on k_gemm_btc
};
ProjPlan plan_projections(const dec_config& c, int rows) {
  ProjPlan pl;
  const bool tc_rows = rows >= 2 && rows <= q4tc_max_tokens() && c.hidden >= 2048;
  const bool q4 = c.linear_fmt == DEC_W_AFFINE4_G64;
  pl.q4tc_all = tc_rows && q4 && c.proj_kernels == DEC_PROJ_TCGEN05;
  pl.q4tc_gu = pl.q4tc_all || (tc_rows && q4 && c.proj_kernels == DEC_PROJ_AUTO && rows >= 16);
  pl.btc = tc_rows && c.linear_fmt == DEC_W_BF16 && c.proj_kernels == DEC_PROJ_TCGEN05;
  return pl;
}

int choose_splits(int N, int K, int fmt, int num_sms) {
  const int cols = fmt == DEC_W_BF16 ? 8 : 16;  // inputs per thread chunk (k_gemv1.cu)
  const int tiles = (N + kGemvRows - 1) / kGemvRows;
  int S = 1;
  while (static_cast<long long>(tiles) * S * 2 < num_sms) {
    const int S2 = S * 2;
    if (K % S2 != 0) break;
    const int KS = K / S2;
    if (KS % cols != 0 || KS / cols < 64) break;
    S = S2;
  }
  return S;
}

// Batched path: inputs staged per chunk (shared-memory bound) and K splits until the grid
// covers the SMs once (bf16) or twice (4-bit, whose CTAs are issue-bound), keeping at
// least 512 (bf16) or 1024 (4-bit) inputs per split: finer splits measured slower, the
// partial-sum round trip (fence, ticket, reload) outweighing the extra CTAs.
void choose_tc_splits(PackedLinear& L, int wfmt, int ny, int num_sms, int tblocks) {
  const int rpb = gemm_tc_rows_per_block(wfmt, ny);
  const int blocks = (L.Npad + rpb - 1) / rpb;
  const int kc_max = gemm_tc_chunk(ny);
  const long long cover = wfmt == kWQ4 ? 2ll * num_sms : num_sms;
  const int min_ks = wfmt == kWQ4 ? 1024 : 512;
  int S = 1;
  // several token blocks already multiply the CTAs (and share one split-K counter set): no split
  while (tblocks == 1 && static_cast<long long>(blocks) * S < cover) {
    const int S2 = S * 2;
    if (L.K % S2 != 0 || (L.K / S2) % kGroup != 0 || L.K / S2 < min_ks) break;
    S = S2;
  }
  L.S = S;
  const int KS = L.K / S;
  int kc = KS;
  for (int div = 1; kc > kc_max || KS % kc != 0 || kc % kGroup != 0; ++div) kc = KS / div;
  L.KC = kc;
}

}  // namespace

// ---------------------------------------------------------------- step enqueue

namespace {

dec_status enqueue_step(dec_handle* h, const StepPtrs& sp, cudaStream_t stream, bool pdl,
                        std::vector<int>* classes) {
  const dec_config& c = h->cfg;
  const int d = c.head_dim, H = c.hidden;
  LaunchCtx lc{stream, false};
  // every launch is an NVTX range named after its kernel class (host-side, around the launch
  // call: a profiler attributes the kernels by range, e.g. ncu --nvtx --nvtx-include "gate_up/");
  // a tool-less process pays a no-op call
  static const char* const kClassNames[DEC_K_COUNT] = {"embed", "qkv", "attention", "o_proj",
                                                       "gate_up", "down", "lm_head"};
  // ranges still open when an error return leaves this function are popped by the guard
  struct NvtxOpen {
    int depth = 0;
    ~NvtxOpen() {
      for (; depth > 0; --depth) nvtxRangePop();
    }
  } nvtx_open;
  auto note = [&](int cls) {
    if (classes) classes->push_back(cls);
    nvtxRangePushA(kClassNames[cls]);
    ++nvtx_open.depth;
  };
  auto check = [&](cudaError_t e, const char* what) -> dec_status {
    if (e != cudaSuccess) {
      set_err("launch of %s failed: %s", what, cudaGetErrorString(e));
      return DEC_ERR_CUDA;
    }
    return DEC_OK;
  };
  // profiling: events around each launch
  int ev = 0;
  auto ev_begin = [&]() -> cudaError_t {
    if (!classes) return cudaSuccess;
    return cudaEventRecord(h->events[2 * ev], stream);
  };
  auto ev_end = [&]() -> cudaError_t {
    if (nvtx_open.depth > 0) {
      nvtxRangePop();
      --nvtx_open.depth;
    }
    if (!classes) return cudaSuccess;
    cudaError_t e = cudaEventRecord(h->events[2 * ev + 1], stream);
    ++ev;
    return e;
  };
  dec_status st;

  EmbedParams ep{};
  ep.embed = h->embed;
  ep.tokens = sp.tokens;
  ep.positions = sp.positions;
  ep.inv_freq = h->inv_freq;
  ep.h = h->h;
  ep.sumsq = h->sumsq;
  ep.rope = h->rope;
  ep.amax_key = h->amax_key;
  ep.status = h->status;
  ep.norm_w0 = h->layers[0].in_norm;
  ep.xhl_out = h->rows > 1 || h->q4tc || h->btc ? h->xh_u : nullptr;
  ep.T = h->tps;
  ep.tl = Timeline{h->timeline, 0};
  ep.V = c.vocab;
  ep.H = H;
  ep.half_d = d / 2;
  ep.max_ctx = c.max_ctx;
  note(DEC_K_EMBED);
  ev_begin();
  if ((st = check(launch_embed(lc, ep, h->rows), "embed")) != DEC_OK) return st;
  ev_end();
  lc.pdl = pdl;

  int launched = 1;  // the embedding kernel
  auto limit_hit = [&]() { return h->launch_limit >= 0 && launched >= h->launch_limit; };
  if (limit_hit()) return DEC_OK;
  // the K/V prefetch of the next GEMV launch (set around the QKV projection only)
  const int kv_elem = c.kv_fmt == DEC_KV_AFFINE8_G64 ? 1 : 2;  // bytes per cached element
  struct {
    const unsigned char* kv = nullptr;
    unsigned long long plane_bytes = 0;
  } kv_pf;
  // x, norm_w: the batch-1 input; xin, xout, next_norm: the batched path's hi/lo planes
  auto gemv = [&](const PackedLinear& L, int in_mode, int epi, const float* x, const __nv_bfloat16* norm_w,
                  float* out, int cls, const char* what, const __nv_bfloat16* xin, __nv_bfloat16* xout,
                  const __nv_bfloat16* next_norm) -> dec_status {
    if (limit_hit()) return DEC_OK;
    ++launched;
    GemvParams gp{};
    gp.w = L.w;
    gp.sb = L.sb;
    gp.N = L.N;
    gp.K = L.K;
    gp.S = L.S;
    gp.KS = L.K / L.S;
    gp.x = x;
    gp.norm_w = norm_w;
    gp.sumsq_in = h->sumsq;
    gp.n_sumsq_in = H / kResGroup;
    gp.eps = c.rms_eps;
    gp.out = out;
    gp.sumsq_out = h->sumsq;
    gp.partials = h->gemv_partials;
    gp.counters = h->gemv_counters;
    gp.amax_key = h->amax_key;
    gp.argmax_out = sp.argmax;
    gp.tl = Timeline{h->timeline, launched - 1};
    if (kv_pf.kv) {
      gp.pf_kv = kv_pf.kv;
      gp.pf_positions = sp.positions;
      gp.pf_plane_bytes = kv_pf.plane_bytes;
      gp.pf_head_bytes = static_cast<unsigned long long>(c.max_ctx) * d * kv_elem;
      gp.pf_B = c.batch;
      gp.pf_nkv = c.n_kv_heads;
      gp.pf_row_bytes = d * kv_elem;
      gp.pf_max_ctx = c.max_ctx;
    }
    note(cls);
    ev_begin();
    dec_status s2;
    if (h->umma) {
      UmmaParams up{};
      up.M = h->rows;
      up.N = L.N;
      up.K = L.K;
      up.m_tiles = (h->rows + umma_tokens_per_tile() - 1) / umma_tokens_per_tile();
      up.tile_n = L.tile_n;
      up.persistent = h->num_sms;
      up.sumsq_in = h->sumsq;
      up.n_sumsq_in = H / kResGroup;
      up.eps = c.rms_eps;
      up.out = out;
      up.sumsq_out = h->sumsq;
      up.xhl_out = xout;
      up.next_norm_w = next_norm;
      up.amax_key = h->amax_key;
      up.argmax_out = sp.argmax;
      up.counters = h->gemv_counters;
      up.status = h->status;
      const void* mx = xin == h->xh_u ? h->map_u : xin == h->xh_o ? h->map_o : h->map_g;
      s2 = check(launch_gemm_umma(lc, mx, L.tmap, up, in_mode, epi), what);
    } else if (L.q4tc || h->btc) {
      Q4tcParams qp{};
      qp.M = h->rows;
      qp.N = L.N;
      qp.K = L.K;
      qp.S = L.S;
      qp.ctas = h->num_sms;
      qp.sb = L.sb;
      qp.sumsq_in = h->sumsq;
      qp.n_sumsq_in = H / kResGroup;
      qp.eps = c.rms_eps;
      qp.out = out;
      qp.sumsq_out = h->sumsq;
      qp.xhl_out = xout;
      qp.next_norm_w = next_norm;
      qp.partials = h->gemv_partials;
      qp.counters = h->gemv_counters;
      qp.amax_key = h->amax_key;
      qp.argmax_out = sp.argmax;
      qp.status = h->status;
      qp.tl = gp.tl;
      qp.pf_kv = gp.pf_kv;  // batch 1: the QKV launch prefetches the attention's K/V (as the GEMV does)
      qp.pf_positions = gp.pf_positions;
      qp.pf_plane_bytes = gp.pf_plane_bytes;
      qp.pf_head_bytes = gp.pf_head_bytes;
      qp.pf_B = gp.pf_B;
      qp.pf_nkv = gp.pf_nkv;
      qp.pf_row_bytes = gp.pf_row_bytes;
      qp.pf_max_ctx = gp.pf_max_ctx;
      const void* mx = xin == h->xh_u ? h->map_u : xin == h->xh_o ? h->map_o : h->map_g;
      s2 = check(L.q4tc ? launch_gemm_q4tc(lc, mx, L.tmap, qp, in_mode, epi)
                         : launch_gemm_btc(lc, mx, L.tmap, qp, in_mode, epi),
                 what);
    } else if (h->rows == 1) {
      s2 = check(launch_gemv1(lc, gp, h->wfmt, in_mode, epi), what);
    } else {
      GemmParams tp{};
      tp.w = L.w;
      tp.N = L.N;
      tp.Npad = L.Npad;
      tp.K = L.K;
      tp.S = L.S;
      tp.KS = L.K / L.S;
      tp.KC = L.KC;
      tp.B = h->rows;
      tp.tblocks = h->tblocks;
      tp.xhl = xin;
      tp.xhl_out = xout;
      tp.next_norm_w = next_norm;
      tp.sumsq_in = h->sumsq;
      tp.n_sumsq_in = H / kResGroup;
      tp.eps = c.rms_eps;
      tp.out = out;
      tp.sumsq_out = h->sumsq;
      tp.partials = h->gemv_partials;
      tp.counters = h->gemv_counters;
      tp.amax_key = h->amax_key;
      tp.argmax_out = sp.argmax;
      tp.tl = gp.tl;
      s2 = check(launch_gemm_tc(lc, tp, h->wfmt, in_mode, epi), what);
    }
    ev_end();
    return s2;
  };

  for (int l = 0; l < c.n_layers; ++l) {
    const PackedLayer& L = h->layers[l];
    if (h->kv_prefetch) {  // bf16 rows, or the codes of the affine 8-bit cache
      const unsigned long long plane =
          static_cast<unsigned long long>(c.batch) * c.n_kv_heads * c.max_ctx * d * kv_elem;
      kv_pf.kv = static_cast<const unsigned char*>(sp.kv) + 2ull * l * plane;
      kv_pf.plane_bytes = plane;
    }
    if ((st = gemv(L.qkv, kInNorm, kEpiStore, h->h, L.in_norm, h->qkv, DEC_K_QKV, "qkv", h->xh_u, nullptr,
                   nullptr)) != DEC_OK)
      return st;
    kv_pf.kv = nullptr;

    AttnParams ap{};
    ap.qkv = h->qkv;
    ap.q_norm = L.q_norm;
    ap.k_norm = L.k_norm;
    ap.rope = h->rope;
    ap.positions = sp.positions;
    attn_set_cache(ap, c, sp.kv);
    ap.layer = l;
    ap.B = h->rows;
    ap.T = h->tps;
    ap.nq = c.n_q_heads;
    ap.nkv = c.n_kv_heads;
    ap.max_ctx = c.max_ctx;
    ap.eps = c.rms_eps;
    ap.out = h->attn_o;
    ap.status = h->status;
    ap.out_hl = h->rows > 1 || h->q4tc || h->btc ? h->xh_o : nullptr;
    if (h->tps > 1) {
      // verify step: every row's K/V go into the cache before any row attends, so
      // that row (b, t) sees the rows (b, 0..t-1) of this step
      if (limit_hit()) return DEC_OK;
      ++launched;
      ap.tl = Timeline{h->timeline, launched - 1};
      note(DEC_K_ATTN);
      ev_begin();
      if ((st = check(launch_kv_append(lc, ap, d), "kv append")) != DEC_OK) return st;
      ev_end();
    }
    if (limit_hit()) return DEC_OK;
    ++launched;
    ap.tl = Timeline{h->timeline, launched - 1};
    note(DEC_K_ATTN);
    ev_begin();
    if ((st = check(h->attn_prefill ? launch_attn_prefill(lc, ap, d) : launch_attention(lc, ap, d), "attention")) !=
        DEC_OK)
      return st;
    ev_end();

    const __nv_bfloat16* after = (l + 1 < c.n_layers) ? h->layers[l + 1].in_norm : h->final_norm;
    if ((st = gemv(L.o, kInPlain, kEpiResid, h->attn_o, nullptr, h->h, DEC_K_OPROJ, "o_proj", h->xh_o, h->xh_u,
                   L.post_norm)) != DEC_OK)
      return st;
    if ((st = gemv(L.gateup, kInNorm, kEpiSwiglu, h->h, L.post_norm, h->g, DEC_K_GATEUP, "gate_up", h->xh_u,
                   h->xh_g, nullptr)) != DEC_OK)
      return st;
    if ((st = gemv(L.down, kInPlain, kEpiResid, h->g, nullptr, h->h, DEC_K_DOWN, "down", h->xh_g, h->xh_u, after)) !=
        DEC_OK)
      return st;
  }
  if ((st = gemv(h->lm_head, kInNorm, kEpiLmHead, h->h, h->final_norm, sp.logits, DEC_K_LMHEAD, "lm_head",
                 h->xh_u, nullptr, nullptr)) != DEC_OK)
    return st;
  return DEC_OK;
}

void drop_one_graph(cudaGraph_t& graph, cudaGraphExec_t& exec, bool& have) {
  if (exec) cudaGraphExecDestroy(exec);
  if (graph) cudaGraphDestroy(graph);
  exec = nullptr;
  graph = nullptr;
  have = false;
}

void drop_graph(dec_handle* h) {
  drop_one_graph(h->graph, h->exec, h->have_graph);
  drop_one_graph(h->hgraph, h->hexec, h->have_hgraph);
}

// The host-staged step's copies: inputs in (tokens and positions are adjacent), argmax out.
dec_status enqueue_io_in(dec_handle* h, cudaStream_t s) {
  DEC_CUDA(cudaMemcpyAsync(h->io_dev, h->io_host, static_cast<size_t>(h->rows + h->cfg.batch) * 4,
                           cudaMemcpyHostToDevice, s));
  return DEC_OK;
}
dec_status enqueue_io_out(dec_handle* h, cudaStream_t s) {
  const size_t off = static_cast<size_t>(h->rows) + h->cfg.batch;
  DEC_CUDA(cudaMemcpyAsync(h->io_host + off, h->io_dev + off, static_cast<size_t>(h->rows) * 4,
                           cudaMemcpyDeviceToHost, s));
  return DEC_OK;
}

// Capture the step for the pointer set sp (with the staging copies around it when `io`) into
// graph / exec.
dec_status capture_into(dec_handle* h, const StepPtrs& sp, bool io, cudaGraph_t& graph_out, cudaGraphExec_t& exec_out,
                        bool& have) {
  drop_one_graph(graph_out, exec_out, have);
  DEC_CUDA(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
  dec_status st = io ? enqueue_io_in(h, h->cap_stream) : DEC_OK;
  if (st == DEC_OK) st = enqueue_step(h, sp, h->cap_stream, true, nullptr);
  if (st == DEC_OK && io) st = enqueue_io_out(h, h->cap_stream);
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(h->cap_stream, &graph);
  if (st != DEC_OK) {
    if (graph) cudaGraphDestroy(graph);
    return st;
  }
  if (e != cudaSuccess) {
    set_err("cudaStreamEndCapture failed: %s", cudaGetErrorString(e));
    return DEC_ERR_CUDA;
  }
  graph_out = graph;
  e = cudaGraphInstantiateWithFlags(&exec_out, graph, 0);
  if (e != cudaSuccess) {
    set_err("cudaGraphInstantiate failed: %s", cudaGetErrorString(e));
    drop_one_graph(graph_out, exec_out, have);
    return DEC_ERR_CUDA;
  }
  have = true;
  return DEC_OK;
}

dec_status capture_graph(dec_handle* h, const StepPtrs& sp) {
  const dec_status st = capture_into(h, sp, false, h->graph, h->exec, h->have_graph);
  if (st == DEC_OK) h->captured = sp;
  return st;
}

dec_status check_step_args(dec_handle* h, const StepPtrs& sp) {
  if (!h) {
    set_err("handle is NULL");
    return DEC_ERR_INVALID_ARG;
  }
  if (!sp.tokens || !sp.positions || !sp.kv || !sp.argmax) {
    set_err("token_ids, positions, kv_cache and argmax_out must be non-NULL");
    return DEC_ERR_INVALID_ARG;
  }
  if (!aligned16(sp.kv)) {
    set_err("kv_cache must be 16-byte aligned");
    return DEC_ERR_INVALID_ARG;
  }
  return DEC_OK;
}

}  // namespace

// ---------------------------------------------------------------- public API

extern "C" size_t dec_kv_cache_bytes(const dec_config* cfg) {
  if (!cfg || cfg->n_layers < 1 || cfg->batch < 1 || cfg->n_kv_heads < 1 || cfg->max_ctx < 1 || cfg->head_dim < 1)
    return 0;
  const size_t rows = static_cast<size_t>(cfg->n_layers) * 2 * cfg->batch * cfg->n_kv_heads * cfg->max_ctx;
  if (cfg->kv_fmt == DEC_KV_BF16) return rows * cfg->head_dim * 2;
  if (cfg->kv_fmt == DEC_KV_AFFINE8_G64 && cfg->head_dim % 64 == 0)
    return kv_q8_params_offset(*cfg) + rows * (cfg->head_dim / 64) * 4;
  return 0;
}

extern "C" const char* dec_last_error(void) { return g_err; }

extern "C" dec_handle* dec_create(const dec_config* cfg, const dec_weights* wts) {
  g_err[0] = 0;
  if (validate(cfg) != DEC_OK) return nullptr;
  if (!wts || !wts->layers || !wts->embed || !wts->final_norm) {
    set_err("weights, weights->layers, embed and final_norm must be non-NULL");
    return nullptr;
  }
  const dec_config c = *cfg;
  const int fmt = c.linear_fmt;
  const int H = c.hidden, d = c.head_dim, nq = c.n_q_heads, nkv = c.n_kv_heads, I = c.intermediate, V = c.vocab;
  if (check_linear(wts->lm_head, fmt, "lm_head", -1) != DEC_OK || !aligned16(wts->embed)) return nullptr;
  for (int l = 0; l < c.n_layers; ++l) {
    const dec_layer_weights& lw = wts->layers[l];
    if (!lw.in_norm || !lw.post_norm || !lw.q_norm || !lw.k_norm) {
      set_err("layer %d: norm weight pointer is NULL", l);
      return nullptr;
    }
    const dec_linear* lins[7] = {&lw.q, &lw.k, &lw.v, &lw.o, &lw.gate, &lw.up, &lw.down};
    const char* names[7] = {"q", "k", "v", "o", "gate", "up", "down"};
    for (int i = 0; i < 7; ++i)
      if (check_linear(*lins[i], fmt, names[i], l) != DEC_OK) return nullptr;
  }

  dec_handle* h = new dec_handle();
  h->cfg = c;
  h->tps = c.tokens_per_seq > 1 ? c.tokens_per_seq : 1;
  h->rows = c.batch * h->tps;
  h->wfmt = fmt == DEC_W_BF16 ? kWBf16 : kWQ4;
  auto fail = [&](const char* what, cudaError_t e) -> dec_handle* {
    set_err("%s: %s", what, cudaGetErrorString(e));
    dec_destroy(h);
    return nullptr;
  };
  cudaError_t e;
  if ((e = cudaGetDevice(&h->device)) != cudaSuccess) return fail("cudaGetDevice", e);
  if ((e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device)) != cudaSuccess)
    return fail("cudaDeviceGetAttribute", e);
  if ((e = cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking)) != cudaSuccess)
    return fail("cudaStreamCreate", e);
  {
    int l2 = 0;
    if ((e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, h->device)) != cudaSuccess)
      return fail("cudaDeviceGetAttribute", e);
    // (the affine 8-bit cache prefetches its codes only)
    const double kv_layer = 2.0 * c.batch * c.n_kv_heads * static_cast<double>(c.max_ctx) * c.head_dim *
                            (c.kv_fmt == DEC_KV_AFFINE8_G64 ? 1 : 2);
    h->kv_prefetch = h->rows == 1 && kv_layer <= l2 / 4.0;
  }

  // ---- packed weight memory
  const int nqkv = (nq + 2 * nkv) * d;
  // the projections' kernel families (plan_projections)
  const ProjPlan pplan = plan_projections(c, h->rows);
  const bool q4tc_all = pplan.q4tc_all, q4tc_gu = pplan.q4tc_gu;
  h->q4tc = q4tc_gu;  // some projection runs on k_gemm_q4tc
  h->btc = pplan.btc;
  const bool tc = h->rows > 1 || h->q4tc || h->btc;
  // more rows than one CTA takes: token blocks of gemm_tc_block_tokens() rows each
  const int blk_tok = gemm_tc_block_tokens(h->wfmt);
  h->tblocks = h->rows > blk_tok ? (h->rows + blk_tok - 1) / blk_tok : 1;
  const int ny = tc ? gemm_tc_ny(h->wfmt, h->rows > blk_tok ? blk_tok : h->rows) : 0;
  // tcgen05 projections for chunks of 128+ rows with bf16 weights on models of hidden >= 2048;
  // below that (the 0.6B shapes) the token-blocked mma.sync kernel's many small CTAs fill the
  // GPU better (512-token chunk: 14.2 ms against 16.2 ms, measured)
  h->umma = h->rows >= umma_tokens_per_tile() && fmt == DEC_W_BF16 && H >= 2048;
  // fragment-packed weights for the mma.sync path, per projection
  auto is_frag = [&](bool on_q4tc) { return tc && !h->umma && !on_q4tc && !h->btc; };
  bool any_frag = false;
  auto lbytes = [&](int N, int K, bool on_q4tc) {
    return is_frag(on_q4tc) ? linear_bytes_tc(fmt, N, K) : linear_bytes(fmt, N, K);
  };
  size_t total = align_up(static_cast<size_t>(V) * H * 2, 256) + align_up(static_cast<size_t>(H) * 2, 256) +
                 lbytes(V, H, q4tc_gu);
  const size_t per_layer = 2 * align_up(static_cast<size_t>(H) * 2, 256) + 2 * align_up(static_cast<size_t>(d) * 2, 256) +
                           lbytes(nqkv, H, q4tc_all) + lbytes(H, nq * d, q4tc_all) + lbytes(2 * I, H, q4tc_gu) +
                           lbytes(H, I, q4tc_all);
  total += per_layer * c.n_layers;
  if ((e = cudaMalloc(&h->wmem, total)) != cudaSuccess) {
    set_err("cudaMalloc of %zu bytes of packed weights failed: %s", total, cudaGetErrorString(e));
    dec_destroy(h);
    return nullptr;
  }
  h->wbytes = total;
  unsigned char* cur = h->wmem;
  auto take = [&](size_t bytes) {
    unsigned char* p = cur;
    cur += align_up(bytes, 256);
    return p;
  };
  auto take_linear = [&](int N, int K, bool on_q4tc) {
    PackedLinear L;
    L.N = N;
    L.K = K;
    L.q4tc = on_q4tc;
    L.frag = is_frag(on_q4tc);
    any_frag = any_frag || L.frag;
    if (L.frag) {
      L.Npad = (N + 15) / 16 * 16;
      choose_tc_splits(L, h->wfmt, ny, h->num_sms, h->tblocks);
      L.w_bytes = linear_bytes_tc(fmt, N, K);
      L.w = take(L.w_bytes);
      return L;
    }
    // (the stream-K bf16 kernel: S = the partial slots its schedule needs)
    L.S = h->umma ? 1
          : L.q4tc ? q4tc_splits(N, K, h->num_sms)
          : h->btc ? btc_max_segments(N, K, h->num_sms)
                   : choose_splits(N, K, fmt, h->num_sms);
    if (fmt == DEC_W_BF16) {
      L.w_bytes = static_cast<size_t>(N) * K * 2;
      L.w = take(L.w_bytes);
    } else {
      L.w_bytes = static_cast<size_t>(N) * K / 2;
      L.sb_bytes = static_cast<size_t>(N) * (K / kGroup) * 4;
      L.w = take(L.w_bytes);
      L.sb = reinterpret_cast<uint32_t*>(take(L.sb_bytes));
    }
    return L;
  };
  h->embed = reinterpret_cast<__nv_bfloat16*>(take(static_cast<size_t>(V) * H * 2));
  h->final_norm = reinterpret_cast<__nv_bfloat16*>(take(static_cast<size_t>(H) * 2));
  h->lm_head = take_linear(V, H, q4tc_gu);
  h->layers.resize(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    PackedLayer& L = h->layers[l];
    L.in_norm = reinterpret_cast<__nv_bfloat16*>(take(static_cast<size_t>(H) * 2));
    L.post_norm = reinterpret_cast<__nv_bfloat16*>(take(static_cast<size_t>(H) * 2));
    L.q_norm = reinterpret_cast<__nv_bfloat16*>(take(static_cast<size_t>(d) * 2));
    L.k_norm = reinterpret_cast<__nv_bfloat16*>(take(static_cast<size_t>(d) * 2));
    L.qkv = take_linear(nqkv, H, q4tc_all);
    L.o = take_linear(H, nq * d, q4tc_all);
    L.gateup = take_linear(2 * I, H, q4tc_gu);
    L.down = take_linear(H, I, q4tc_all);
  }

  // ---- pack (device to device on the internal stream)
  cudaStream_t s = h->cap_stream;
  auto cp = [&](void* dst, const void* src, size_t bytes) { return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s); };
  auto pack_lin = [&](const PackedLinear& P, size_t row_off, const dec_linear& a, const dec_linear* b, int rows,
                      int K, int ib) -> cudaError_t {
    if (P.frag) {
      const int npad = (rows + 15) / 16 * 16;
      if (fmt == DEC_W_BF16)
        return pack_frag_bf16(s, static_cast<uint32_t*>(P.w), static_cast<const __nv_bfloat16*>(a.w),
                              b ? static_cast<const __nv_bfloat16*>(b->w) : nullptr, rows, npad, K, ib,
                              static_cast<int>(row_off), npad);
      return pack_frag_q4(s, static_cast<unsigned char*>(P.w), static_cast<const uint32_t*>(a.w),
                          static_cast<const __nv_bfloat16*>(a.scales), static_cast<const __nv_bfloat16*>(a.biases),
                          b ? static_cast<const uint32_t*>(b->w) : nullptr,
                          b ? static_cast<const __nv_bfloat16*>(b->scales) : nullptr,
                          b ? static_cast<const __nv_bfloat16*>(b->biases) : nullptr, rows, K, ib,
                          static_cast<int>(row_off), npad);
    }
    if (fmt == DEC_W_BF16) {
      return pack_rows_bf16(s, static_cast<__nv_bfloat16*>(P.w) + row_off * K, static_cast<const __nv_bfloat16*>(a.w),
                            b ? static_cast<const __nv_bfloat16*>(b->w) : nullptr, rows, K, ib);
    }
    return pack_rows_q4(s, static_cast<uint32_t*>(P.w) + row_off * (K / 8), P.sb + row_off * (K / kGroup),
                        static_cast<const uint32_t*>(a.w), static_cast<const __nv_bfloat16*>(a.scales),
                        static_cast<const __nv_bfloat16*>(a.biases), b ? static_cast<const uint32_t*>(b->w) : nullptr,
                        b ? static_cast<const __nv_bfloat16*>(b->scales) : nullptr,
                        b ? static_cast<const __nv_bfloat16*>(b->biases) : nullptr, rows, K, ib);
  };
  if ((e = cp(h->embed, wts->embed, static_cast<size_t>(V) * H * 2)) != cudaSuccess) return fail("copy embed", e);
  if ((e = cp(h->final_norm, wts->final_norm, static_cast<size_t>(H) * 2)) != cudaSuccess) return fail("copy norm", e);
  if ((e = pack_lin(h->lm_head, 0, wts->lm_head, nullptr, V, H, 0)) != cudaSuccess) return fail("pack lm_head", e);
  for (int l = 0; l < c.n_layers; ++l) {
    const dec_layer_weights& lw = wts->layers[l];
    PackedLayer& L = h->layers[l];
    if ((e = cp(L.in_norm, lw.in_norm, static_cast<size_t>(H) * 2)) != cudaSuccess) return fail("copy norm", e);
    if ((e = cp(L.post_norm, lw.post_norm, static_cast<size_t>(H) * 2)) != cudaSuccess) return fail("copy norm", e);
    if ((e = cp(L.q_norm, lw.q_norm, static_cast<size_t>(d) * 2)) != cudaSuccess) return fail("copy norm", e);
    if ((e = cp(L.k_norm, lw.k_norm, static_cast<size_t>(d) * 2)) != cudaSuccess) return fail("copy norm", e);
    if ((e = pack_lin(L.qkv, 0, lw.q, nullptr, nq * d, H, 0)) != cudaSuccess) return fail("pack q", e);
    if ((e = pack_lin(L.qkv, static_cast<size_t>(nq) * d, lw.k, nullptr, nkv * d, H, 0)) != cudaSuccess)
      return fail("pack k", e);
    if ((e = pack_lin(L.qkv, static_cast<size_t>(nq + nkv) * d, lw.v, nullptr, nkv * d, H, 0)) != cudaSuccess)
      return fail("pack v", e);
    if ((e = pack_lin(L.o, 0, lw.o, nullptr, H, nq * d, 0)) != cudaSuccess) return fail("pack o", e);
    if ((e = pack_lin(L.gateup, 0, lw.gate, &lw.up, 2 * I, H, h->umma ? 16 : L.gateup.frag ? 8 : kGemvRows / 2)) !=
        cudaSuccess)
      return fail("pack gate/up", e);
    if ((e = pack_lin(L.down, 0, lw.down, nullptr, H, I, 0)) != cudaSuccess) return fail("pack down", e);
  }

  const int G = nq / nkv;
  // ---- workspace (one row per token of the step)
  const int B = h->rows;
  int max_tiles = 0;
  size_t max_partials = 0;
  auto acc_lin = [&](const PackedLinear& L) {
    const int tiles = (L.N + kGemvRows - 1) / kGemvRows;  // >= row blocks of the batched path too
    max_tiles = tiles > max_tiles ? tiles : max_tiles;
    if (L.S > 1) {
      const size_t pp =
          L.frag ? static_cast<size_t>(L.S) * (L.Npad / 16) * 32 * ny * 4 : static_cast<size_t>(L.S) * L.N * B;
      max_partials = pp > max_partials ? pp : max_partials;
    }
  };
  acc_lin(h->lm_head);
  for (auto& L : h->layers) {
    acc_lin(L.qkv);
    acc_lin(L.o);
    acc_lin(L.gateup);
    acc_lin(L.down);
  }
  size_t ws_bytes = 0;
  auto plan = [&](size_t bytes) {
    size_t off = ws_bytes;
    ws_bytes += align_up(bytes, 256);
    return off;
  };
  const size_t o_h = plan(static_cast<size_t>(B) * H * 4);
  const size_t o_qkv = plan(static_cast<size_t>(B) * nqkv * 4);
  const size_t o_att = plan(static_cast<size_t>(B) * nq * d * 4);
  const size_t o_g = plan(static_cast<size_t>(B) * I * 4);
  const size_t o_ss = plan(static_cast<size_t>(B) * (H / kResGroup) * 4);
  const size_t o_xu = plan(static_cast<size_t>(2) * B * H * 2);
  const size_t o_xo = plan(static_cast<size_t>(2) * B * nq * d * 2);
  const size_t o_xg = plan(static_cast<size_t>(2) * B * I * 2);
  const size_t o_gp = plan((max_partials ? max_partials : 1) * 4);
  const size_t o_gc = plan((static_cast<size_t>(max_tiles) * h->tblocks + 1) * 4);
  const size_t o_rope = plan(static_cast<size_t>(B) * (d / 2) * 8);
  const size_t o_inv = plan(static_cast<size_t>(d / 2) * 8);
  const size_t o_key = plan(static_cast<size_t>(B) * 8);
  const size_t o_st = plan(4);
  if ((e = cudaMalloc(&h->ws, ws_bytes)) != cudaSuccess) {
    set_err("cudaMalloc of %zu bytes of workspace failed: %s", ws_bytes, cudaGetErrorString(e));
    dec_destroy(h);
    return nullptr;
  }
  if ((e = cudaMemsetAsync(h->ws, 0, ws_bytes, s)) != cudaSuccess) return fail("memset workspace", e);
  h->h = reinterpret_cast<float*>(h->ws + o_h);
  h->qkv = reinterpret_cast<float*>(h->ws + o_qkv);
  h->attn_o = reinterpret_cast<float*>(h->ws + o_att);
  h->g = reinterpret_cast<float*>(h->ws + o_g);
  h->sumsq = reinterpret_cast<float*>(h->ws + o_ss);
  h->xh_u = reinterpret_cast<__nv_bfloat16*>(h->ws + o_xu);
  h->xh_o = reinterpret_cast<__nv_bfloat16*>(h->ws + o_xo);
  h->xh_g = reinterpret_cast<__nv_bfloat16*>(h->ws + o_xg);
  h->gemv_partials = reinterpret_cast<float*>(h->ws + o_gp);
  h->gemv_counters = reinterpret_cast<unsigned*>(h->ws + o_gc);
  h->rope = reinterpret_cast<float2*>(h->ws + o_rope);
  h->inv_freq = reinterpret_cast<double*>(h->ws + o_inv);
  h->amax_key = reinterpret_cast<unsigned long long*>(h->ws + o_key);
  h->status = reinterpret_cast<unsigned*>(h->ws + o_st);

  // RoPE inverse frequencies theta^(-2i/d), i < d/2, in double on the host
  std::vector<double> inv(d / 2);
  for (int i = 0; i < d / 2; ++i) inv[i] = std::pow(static_cast<double>(c.rope_theta), -2.0 * i / d);
  if ((e = cudaMemcpyAsync(h->inv_freq, inv.data(), inv.size() * 8, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return fail("upload inv_freq", e);
  if ((e = prepare_attention(d, G, c.kv_fmt)) != cudaSuccess) return fail("attention kernel attributes", e);
  h->attn_prefill = h->tps >= attn_prefill_min_tokens() && c.kv_fmt == DEC_KV_BF16;
  if (h->attn_prefill && (e = prepare_attn_prefill(d, G)) != cudaSuccess)
    return fail("prefill attention kernel attributes", e);
  if (h->umma) {  // tensor maps of every weight and of the activation planes, kernel attributes
    auto lmap = [&](PackedLinear& L) {
      L.tile_n = umma_tile_n(h->rows, L.N, h->num_sms);
      return umma_tensor_map(L.tmap, L.w, L.N, L.K, L.tile_n);
    };
    if ((e = lmap(h->lm_head)) != cudaSuccess) return fail("tensor map", e);
    for (auto& L : h->layers)
      if ((e = lmap(L.qkv)) != cudaSuccess || (e = lmap(L.o)) != cudaSuccess || (e = lmap(L.gateup)) != cudaSuccess ||
          (e = lmap(L.down)) != cudaSuccess)
        return fail("tensor map", e);
    const int tok = umma_tokens_per_tile();
    if ((e = umma_tensor_map(h->map_u, h->xh_u, 2 * h->rows, H, tok)) != cudaSuccess ||
        (e = umma_tensor_map(h->map_o, h->xh_o, 2 * h->rows, nq * d, tok)) != cudaSuccess ||
        (e = umma_tensor_map(h->map_g, h->xh_g, 2 * h->rows, I, tok)) != cudaSuccess)
      return fail("tensor map", e);
    const int combos[4][2] = {{kInNorm, kEpiStore}, {kInPlain, kEpiResid}, {kInNorm, kEpiSwiglu}, {kInNorm, kEpiLmHead}};
    for (auto& cb : combos)
      for (int tn : {128, 256})
        if ((e = prepare_gemm_umma(cb[0], cb[1], tn)) != cudaSuccess) return fail("tcgen05 kernel attributes", e);
  }
  if (h->q4tc || h->btc) {  // TMA maps of their weights and of the activation planes, kernel attributes
    auto cmap = [&](PackedLinear& L) {
      return L.q4tc ? q4tc_code_map(L.tmap, L.w, L.N, L.K)
             : h->btc ? umma_tensor_map(L.tmap, L.w, L.N, L.K, 128)
                      : cudaSuccess;
    };
    if ((e = cmap(h->lm_head)) != cudaSuccess) return fail("tensor map", e);
    for (auto& L : h->layers)
      if ((e = cmap(L.qkv)) != cudaSuccess || (e = cmap(L.o)) != cudaSuccess || (e = cmap(L.gateup)) != cudaSuccess ||
          (e = cmap(L.down)) != cudaSuccess)
        return fail("tensor map", e);
    const int tok = h->q4tc ? q4tc_max_tokens() : btc_box_rows(h->rows);
    if ((e = umma_tensor_map(h->map_u, h->xh_u, 2 * h->rows, H, tok)) != cudaSuccess ||
        (e = umma_tensor_map(h->map_o, h->xh_o, 2 * h->rows, nq * d, tok)) != cudaSuccess ||
        (e = umma_tensor_map(h->map_g, h->xh_g, 2 * h->rows, I, tok)) != cudaSuccess)
      return fail("tensor map", e);
    const int combos[4][2] = {{kInNorm, kEpiStore}, {kInPlain, kEpiResid}, {kInNorm, kEpiSwiglu}, {kInNorm, kEpiLmHead}};
    for (auto& cb : combos)
      if ((e = h->q4tc ? prepare_gemm_q4tc(cb[0], cb[1]) : prepare_gemm_btc(cb[0], cb[1])) != cudaSuccess)
        return fail("tcgen05 decode kernel attributes", e);
  }
  if (any_frag) {
    GemmParams gp{};
    gp.B = h->rows;
    gp.tblocks = h->tblocks;
    gp.KC = gemm_tc_chunk(ny);
    const int combos[4][2] = {{kInNorm, kEpiStore}, {kInPlain, kEpiResid}, {kInNorm, kEpiSwiglu}, {kInNorm, kEpiLmHead}};
    for (auto& cb : combos)
      if ((e = prepare_gemm_tc(gp, h->wfmt, cb[0], cb[1])) != cudaSuccess) return fail("batched kernel attributes", e);
  }
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail("packing", e);
  return h;
}

extern "C" void dec_destroy(dec_handle* h) {
  if (!h) return;
  drop_graph(h);
  for (cudaEvent_t ev : h->events) cudaEventDestroy(ev);
  if (h->hold_ev) cudaEventDestroy(h->hold_ev);
  if (h->hold_stream) cudaStreamDestroy(h->hold_stream);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->io_host) cudaFreeHost(h->io_host);
  if (h->io_dev) cudaFree(h->io_dev);
  if (h->wmem) cudaFree(h->wmem);
  if (h->ws) cudaFree(h->ws);
  delete h;
}

extern "C" dec_status dec_step(dec_handle* h, const int32_t* token_ids, const int32_t* positions, void* kv_cache,
                               float* logits_out, int32_t* argmax_out, dec_stream_t stream) {
  const StepPtrs sp{token_ids, positions, kv_cache, logits_out, argmax_out};
  dec_status st = check_step_args(h, sp);
  if (st != DEC_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (!h->graph_mode) {
    st = enqueue_step(h, sp, cs, true, nullptr);
    return st;
  }
  if (!h->have_graph || !(h->captured == sp)) {
    if ((st = capture_graph(h, sp)) != DEC_OK) return st;
  }
  DEC_CUDA(cudaGraphLaunch(h->exec, cs));
  return DEC_OK;
}

extern "C" dec_status dec_step_host(dec_handle* h, const int32_t* token_ids, const int32_t* positions,
                                    void* kv_cache, float* logits_out, int32_t* argmax_out, dec_stream_t stream) {
  if (!h) {
    set_err("handle is NULL");
    return DEC_ERR_INVALID_ARG;
  }
  if (!token_ids || !positions || !argmax_out) {
    set_err("token_ids, positions and argmax_out must be non-NULL host pointers");
    return DEC_ERR_INVALID_ARG;
  }
  const size_t rows = static_cast<size_t>(h->rows), B = static_cast<size_t>(h->cfg.batch);
  const size_t n_io = 2 * rows + B;
  if (!h->io_host) {
    void* ph = nullptr;
    void* pd = nullptr;
    cudaError_t e = cudaHostAlloc(&ph, n_io * 4, cudaHostAllocDefault);
    if (e == cudaSuccess) e = cudaMalloc(&pd, n_io * 4);
    if (e != cudaSuccess) {
      if (ph) cudaFreeHost(ph);
      set_err("staging buffers for dec_step_host (%zu bytes): %s", n_io * 4, cudaGetErrorString(e));
      return DEC_ERR_OOM;
    }
    h->io_host = static_cast<int32_t*>(ph);
    h->io_dev = static_cast<int32_t*>(pd);
  }
  const StepPtrs sp{h->io_dev, h->io_dev + rows, kv_cache, logits_out, h->io_dev + rows + B};
  dec_status st = check_step_args(h, sp);
  if (st != DEC_OK) return st;
  // inputs into the pinned staging first: argmax_out may alias token_ids
  std::memcpy(h->io_host, token_ids, rows * 4);
  std::memcpy(h->io_host + rows, positions, B * 4);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (!h->graph_mode) {
    if ((st = enqueue_io_in(h, cs)) != DEC_OK) return st;
    if ((st = enqueue_step(h, sp, cs, true, nullptr)) != DEC_OK) return st;
    if ((st = enqueue_io_out(h, cs)) != DEC_OK) return st;
  } else {
    if (!h->have_hgraph || !(h->hcaptured == sp)) {
      if ((st = capture_into(h, sp, true, h->hgraph, h->hexec, h->have_hgraph)) != DEC_OK) return st;
      h->hcaptured = sp;
    }
    DEC_CUDA(cudaGraphLaunch(h->hexec, cs));
  }
  DEC_CUDA(cudaStreamSynchronize(cs));
  std::memcpy(argmax_out, h->io_host + rows + B, rows * 4);
  return DEC_OK;
}

extern "C" dec_status dec_set_graph_mode(dec_handle* h, int enabled) {
  if (!h) {
    set_err("handle is NULL");
    return DEC_ERR_INVALID_ARG;
  }
  h->graph_mode = enabled != 0;
  return DEC_OK;
}

extern "C" dec_status dec_get_device_status(dec_handle* h, int* out) {
  if (!h || !out) {
    set_err("handle and out must be non-NULL");
    return DEC_ERR_INVALID_ARG;
  }
  unsigned v = 0;
  DEC_CUDA(cudaMemcpy(&v, h->status, 4, cudaMemcpyDeviceToHost));
  const unsigned zero = 0;
  DEC_CUDA(cudaMemcpy(h->status, &zero, 4, cudaMemcpyHostToDevice));
  *out = static_cast<int>(v);
  if (v & kStatusTimeout) {
    set_err("a bounded device wait timed out");
    return DEC_ERR_TIMEOUT;
  }
  if (v) {
    set_err("device input out of range (status bits 0x%x)", v);
    return DEC_ERR_DEVICE_INPUT;
  }
  return DEC_OK;
}

namespace {
// rows per gate (then up) block of the packed gate/up projection
int gate_up_block(const dec_handle* h, const PackedLinear& L) {
  return h->umma ? 16 : L.frag ? 8 : kGemvRows / 2;
}
}  // namespace

extern "C" dec_status dec_debug_dequant(dec_handle* h, int layer, int which, float* out, dec_stream_t stream) {
  if (!h || !out || which < 0 || which > 7 || (which < 7 && (layer < 0 || layer >= h->cfg.n_layers))) {
    set_err("dec_debug_dequant: bad arguments");
    return DEC_ERR_INVALID_ARG;
  }
  const dec_config& c = h->cfg;
  const int d = c.head_dim, H = c.hidden;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const PackedLinear* P;
  int rows, K, off = 0, ib = 0, half = -1;
  if (which == 7) {
    P = &h->lm_head;
    rows = c.vocab;
    K = H;
  } else {
    const PackedLayer& L = h->layers[layer];
    switch (which) {
      case 0: P = &L.qkv; rows = c.n_q_heads * d; K = H; break;
      case 1: P = &L.qkv; rows = c.n_kv_heads * d; K = H; off = c.n_q_heads * d; break;
      case 2: P = &L.qkv; rows = c.n_kv_heads * d; K = H; off = (c.n_q_heads + c.n_kv_heads) * d; break;
      case 3: P = &L.o; rows = H; K = c.n_q_heads * d; break;
      case 4: P = &L.gateup; rows = c.intermediate; K = H; ib = gate_up_block(h, L.gateup); half = 0; break;
      case 5: P = &L.gateup; rows = c.intermediate; K = H; ib = gate_up_block(h, L.gateup); half = 1; break;
      default: P = &L.down; rows = H; K = c.intermediate; break;
    }
  }
  if (P->frag) {
    DEC_CUDA(debug_dequant_frag(cs, out, P->w, h->wfmt, rows, K, off, ib, half));
  } else {
    DEC_CUDA(debug_dequant(cs, out, P->w, P->sb, h->wfmt, rows, K, off, ib, half));
  }
  return DEC_OK;
}

extern "C" dec_status dec_debug_force_timeout(dec_handle* h, int polls, dec_stream_t stream) {
  if (!h || polls < 1 || polls > 65536) {
    set_err("dec_debug_force_timeout: handle is NULL or polls outside 1..65536");
    return DEC_ERR_INVALID_ARG;
  }
  DEC_CUDA(launch_force_timeout(reinterpret_cast<cudaStream_t>(stream), h->status, polls));
  return DEC_OK;
}

extern "C" dec_status dec_advance(const int32_t* argmax, int32_t* token_ids, int32_t* positions, int batch,
                                  dec_stream_t stream) {
  if (!argmax || !token_ids || !positions || batch < 1) {
    set_err("dec_advance: bad arguments");
    return DEC_ERR_INVALID_ARG;
  }
  DEC_CUDA(launch_advance(reinterpret_cast<cudaStream_t>(stream), argmax, token_ids, positions, batch));
  return DEC_OK;
}

extern "C" int dec_launches_per_step(const dec_handle* h) {
  return h ? (h->tps > 1 ? 6 : 5) * h->cfg.n_layers + 2 : 0;
}

extern "C" dec_status dec_profile_step(dec_handle* h, const int32_t* token_ids, const int32_t* positions,
                                       void* kv_cache, float* logits_out, int32_t* argmax_out, dec_stream_t stream,
                                       double* ms, int* launches, int n_classes) {
  const StepPtrs sp{token_ids, positions, kv_cache, logits_out, argmax_out};
  dec_status st = check_step_args(h, sp);
  if (st != DEC_OK) return st;
  if (!ms || !launches || n_classes < DEC_K_COUNT) {
    set_err("dec_profile_step: ms/launches must hold DEC_K_COUNT entries");
    return DEC_ERR_INVALID_ARG;
  }
  const int n = dec_launches_per_step(h);
  while (static_cast<int>(h->events.size()) < 2 * n) {
    cudaEvent_t ev;
    DEC_CUDA(cudaEventCreate(&ev));
    h->events.push_back(ev);
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (!h->hold_stream) DEC_CUDA(cudaStreamCreateWithFlags(&h->hold_stream, cudaStreamNonBlocking));
  if (!h->hold_ev) DEC_CUDA(cudaEventCreateWithFlags(&h->hold_ev, cudaEventDisableTiming));
  // about 10 us of host time per launch to enqueue, plus a margin
  DEC_CUDA(launch_hold(h->hold_stream, 200000ull + 10000ull * static_cast<unsigned long long>(n)));
  DEC_CUDA(cudaEventRecord(h->hold_ev, h->hold_stream));
  DEC_CUDA(cudaStreamWaitEvent(cs, h->hold_ev, 0));
  std::vector<int> classes;
  if ((st = enqueue_step(h, sp, cs, false, &classes)) != DEC_OK) return st;
  DEC_CUDA(cudaStreamSynchronize(cs));
  for (size_t i = 0; i < classes.size(); ++i) {
    float t = 0.f;
    DEC_CUDA(cudaEventElapsedTime(&t, h->events[2 * i], h->events[2 * i + 1]));
    ms[classes[i]] += t;
    launches[classes[i]] += 1;
  }
  return DEC_OK;
}

extern "C" double dec_kernel_bytes(const dec_handle* h, int cls, double mean_cached_len) {
  if (!h) return 0.0;
  const dec_config& c = h->cfg;
  const double wb = wbytes_per_elem(c.linear_fmt);
  const double H = c.hidden, d = c.head_dim, nq = c.n_q_heads, nkv = c.n_kv_heads, I = c.intermediate, V = c.vocab;
  const double B = h->rows, T = h->tps;
  switch (cls) {
    case DEC_K_EMBED: return B * H * 2.0;
    case DEC_K_QKV: return (nq + 2 * nkv) * d * H * wb + H * 2.0;
    // every row reads its sequence's slots 0 .. P + t (t < T: its place among the step's rows);
    // a slot is a bf16 row, or a row of codes and a (scale, bias) pair per 64.  The prefill
    // attention reads each sequence's slots 0 .. P + T - 1 once for all of its rows.
    case DEC_K_ATTN: {
      const double row = c.kv_fmt == DEC_KV_AFFINE8_G64 ? d + 4.0 * (d / 64.0) : 2.0 * d;
      if (h->attn_prefill) return (B / T) * nkv * 2.0 * row * (mean_cached_len + T);
      return B * nkv * 2.0 * row * (mean_cached_len + 1.0 + (T - 1.0) / 2.0) + 2.0 * row;
    }
    case DEC_K_OPROJ: return H * nq * d * wb;
    case DEC_K_GATEUP: return 2.0 * I * H * wb + H * 2.0;
    case DEC_K_DOWN: return H * I * wb;
    case DEC_K_LMHEAD: return V * H * wb + H * 2.0;
    default: return 0.0;
  }
}

// ---------------------------------------------------------------- stand-alone attention kernel

namespace {


size_t attention_workspace_total(const dec_config* c) {
  return align_up(static_cast<size_t>(c->batch) * (c->head_dim / 2) * 8, 256);  // RoPE (cos, sin) table
}

}  // namespace

extern "C" size_t dec_attention_workspace_bytes(const dec_config* cfg) {
  if (validate_attention_cfg(cfg, 0) != DEC_OK) return 0;
  return attention_workspace_total(cfg);
}

extern "C" dec_status dec_attention(const dec_config* cfg, int layer, const float* qkv, const void* q_norm,
                                    const void* k_norm, const int32_t* positions, void* kv_cache, float* out,
                                    void* workspace, size_t workspace_bytes, dec_stream_t stream) {
  dec_status st = validate_attention_cfg(cfg, layer);
  if (st != DEC_OK) return st;
  if (!qkv || !q_norm || !k_norm || !positions || !kv_cache || !out || !workspace || !aligned16(kv_cache) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
    set_err("dec_attention: NULL pointer, kv_cache not 16-byte aligned or workspace not 256-byte aligned");
    return DEC_ERR_INVALID_ARG;
  }
  const size_t need = attention_workspace_total(cfg);
  if (workspace_bytes < need) {
    set_err("dec_attention: workspace of %zu bytes, %zu needed", workspace_bytes, need);
    return DEC_ERR_INVALID_ARG;
  }
  const int G = cfg->n_q_heads / cfg->n_kv_heads;
  DEC_CUDA(prepare_attention(cfg->head_dim, G, cfg->kv_fmt));
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  float2* rope = static_cast<float2*>(workspace);
  DEC_CUDA(launch_rope_table(cs, positions, cfg->batch, cfg->head_dim, cfg->max_ctx, cfg->rope_theta, rope, nullptr));
  AttnParams ap{};
  ap.qkv = qkv;
  ap.q_norm = static_cast<const __nv_bfloat16*>(q_norm);
  ap.k_norm = static_cast<const __nv_bfloat16*>(k_norm);
  ap.rope = rope;
  ap.positions = positions;
  attn_set_cache(ap, *cfg, kv_cache);
  ap.layer = layer;
  ap.B = cfg->batch;
  ap.nq = cfg->n_q_heads;
  ap.nkv = cfg->n_kv_heads;
  ap.max_ctx = cfg->max_ctx;
  ap.eps = cfg->rms_eps;
  ap.out = out;
  ap.status = nullptr;
  DEC_CUDA(launch_attention(LaunchCtx{cs, false}, ap, cfg->head_dim));
  return DEC_OK;
}

extern "C" dec_status dec_debug_gemm_tc5(const void* x_hl, int M, const void* w, int N, int K, float* out,
                                         int persistent, dec_stream_t stream) {
  g_err[0] = 0;
  if (!x_hl || !w || !out || M < 1 || N < 1 || K < 64 || K % 64 != 0 || !aligned16(x_hl) || !aligned16(w)) {
    set_err("dec_debug_gemm_tc5: NULL or misaligned pointer, M or N < 1, or K not a positive multiple of 64");
    return DEC_ERR_INVALID_ARG;
  }
  alignas(64) unsigned char mx[128], mw[128];
  int dev = 0, sms = 0;
  DEC_CUDA(cudaGetDevice(&dev));
  DEC_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int tn = umma_tile_n(M, N, sms);
  DEC_CUDA(umma_tensor_map(mx, x_hl, 2 * M, K, umma_tokens_per_tile()));
  DEC_CUDA(umma_tensor_map(mw, w, N, K, tn));
  DEC_CUDA(prepare_gemm_umma(kInPlain, kEpiStore, tn));
  UmmaParams p{};
  p.tile_n = tn;
  p.persistent = persistent ? sms : 0;
  p.M = M;
  p.N = N;
  p.K = K;
  p.m_tiles = (M + umma_tokens_per_tile() - 1) / umma_tokens_per_tile();
  p.out = out;
  DEC_CUDA(launch_gemm_umma(LaunchCtx{reinterpret_cast<cudaStream_t>(stream), false}, mx, mw, p, kInPlain, kEpiStore));
  return DEC_OK;
}

extern "C" dec_status dec_debug_gemm_q4tc(const void* x_hl, int M, const void* codes, const void* sb, int N, int K,
                                          int S, float* out, float* partials, unsigned* counters,
                                          dec_stream_t stream) {
  g_err[0] = 0;
  if (!x_hl || !codes || !sb || !out || M < 1 || M > q4tc_max_tokens() || N < 1 || K < 64 || K % 64 != 0 || S < 1 ||
      (K / 64) % S != 0 || (S > 1 && (!partials || !counters)) || !aligned16(x_hl) || !aligned16(codes) ||
      !aligned16(sb)) {
    set_err("dec_debug_gemm_q4tc: NULL or misaligned pointer, M outside 1..%d, N < 1, K not a positive multiple of "
            "64, or S not dividing K / 64 (S > 1 needs partials and counters)",
            q4tc_max_tokens());
    return DEC_ERR_INVALID_ARG;
  }
  alignas(64) unsigned char mx[128], mc[128];
  int dev = 0, sms = 0;
  DEC_CUDA(cudaGetDevice(&dev));
  DEC_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  DEC_CUDA(umma_tensor_map(mx, x_hl, 2 * M, K, q4tc_max_tokens()));
  DEC_CUDA(q4tc_code_map(mc, codes, N, K));
  DEC_CUDA(prepare_gemm_q4tc(kInPlain, kEpiStore));
  Q4tcParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.S = S;
  p.ctas = sms;
  p.sb = static_cast<const uint32_t*>(sb);
  p.out = out;
  p.partials = partials;
  p.counters = counters;
  DEC_CUDA(launch_gemm_q4tc(LaunchCtx{reinterpret_cast<cudaStream_t>(stream), false}, mx, mc, p, kInPlain, kEpiStore));
  return DEC_OK;
}

extern "C" dec_status dec_debug_gemm_btc(const void* x_hl, int M, const void* w, int N, int K, int ctas, float* out,
                                         float* partials, unsigned* counters, dec_stream_t stream) {
  g_err[0] = 0;
  if (!x_hl || !w || !out || !partials || !counters || M < 1 || M > q4tc_max_tokens() || N < 1 || K < 64 ||
      K % 64 != 0 || !aligned16(x_hl) || !aligned16(w)) {
    set_err("dec_debug_gemm_btc: NULL or misaligned pointer, M outside 1..%d, N < 1, or K not a positive multiple "
            "of 64",
            q4tc_max_tokens());
    return DEC_ERR_INVALID_ARG;
  }
  alignas(64) unsigned char mx[128], mw[128];
  int dev = 0, sms = 0;
  DEC_CUDA(cudaGetDevice(&dev));
  DEC_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  DEC_CUDA(umma_tensor_map(mx, x_hl, 2 * M, K, btc_box_rows(M)));
  DEC_CUDA(umma_tensor_map(mw, w, N, K, 128));
  DEC_CUDA(prepare_gemm_btc(kInPlain, kEpiStore));
  Q4tcParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.S = 1;
  p.ctas = ctas > 0 ? ctas : sms;
  p.out = out;
  p.partials = partials;
  p.counters = counters;
  DEC_CUDA(launch_gemm_btc(LaunchCtx{reinterpret_cast<cudaStream_t>(stream), false}, mx, mw, p, kInPlain, kEpiStore));
  return DEC_OK;
}

extern "C" dec_status dec_debug_proj_plan(const dec_config* cfg, int* tcgen05_mask) {
  g_err[0] = 0;
  if (!cfg || !tcgen05_mask) {
    set_err("dec_debug_proj_plan: NULL argument");
    return DEC_ERR_INVALID_ARG;
  }
  const dec_status st = validate(cfg);
  if (st != DEC_OK) return st;
  const int tps = cfg->tokens_per_seq > 1 ? cfg->tokens_per_seq : 1;
  const ProjPlan pl = plan_projections(*cfg, cfg->batch * tps);
  const bool rest = pl.q4tc_all || pl.btc, gu = pl.q4tc_gu || pl.btc;
  *tcgen05_mask = (rest ? 1 | 2 | 8 : 0) | (gu ? 4 | 16 : 0);
  return DEC_OK;
}

extern "C" int dec_debug_btc_max_segments(int N, int K, int ctas) {
  if (N < 1 || K < 64 || ctas < 1) return 0;
  return btc_max_segments(N, K, ctas);
}

extern "C" dec_status dec_kv_quantize(const float* src, int rows, int head_dim, uint8_t* codes, void* params,
                                      dec_stream_t stream) {
  g_err[0] = 0;
  if (head_dim != 64 && head_dim != 128) {
    set_err("dec_kv_quantize: head_dim must be 64 or 128 (got %d)", head_dim);
    return DEC_ERR_UNSUPPORTED;
  }
  if (rows < 0 || (rows > 0 && (!src || !codes || !params)) ||
      (reinterpret_cast<uintptr_t>(params) & 3u)) {
    set_err("dec_kv_quantize: rows < 0, a NULL buffer, or params not 4-byte aligned");
    return DEC_ERR_INVALID_ARG;
  }
  DEC_CUDA(launch_kv_quantize(reinterpret_cast<cudaStream_t>(stream), src, rows, head_dim, codes,
                              static_cast<__nv_bfloat16*>(params)));
  return DEC_OK;
}

// ---------------------------------------------------------------- debug hooks

extern "C" dec_status dec_debug_step_prefix(dec_handle* h, const int32_t* token_ids, const int32_t* positions,
                                            void* kv_cache, float* logits_out, int32_t* argmax_out,
                                            dec_stream_t stream, int n_launches) {
  const StepPtrs sp{token_ids, positions, kv_cache, logits_out, argmax_out};
  dec_status st = check_step_args(h, sp);
  if (st != DEC_OK) return st;
  if (n_launches < 1) {
    set_err("dec_debug_step_prefix: n_launches must be >= 1");
    return DEC_ERR_INVALID_ARG;
  }
  h->launch_limit = n_launches;
  st = enqueue_step(h, sp, reinterpret_cast<cudaStream_t>(stream), false, nullptr);
  h->launch_limit = -1;
  return st;
}

extern "C" dec_status dec_debug_buffer(dec_handle* h, int which, void* dst, size_t bytes, dec_stream_t stream) {
  if (!h || !dst) {
    set_err("dec_debug_buffer: NULL argument");
    return DEC_ERR_INVALID_ARG;
  }
  const dec_config& c = h->cfg;
  const size_t B = h->rows;
  const void* src = nullptr;
  size_t n = 0;
  switch (which) {
    case 0: src = h->h; n = B * c.hidden * 4; break;
    case 1: src = h->qkv; n = B * (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim * 4; break;
    case 2: src = h->attn_o; n = B * c.n_q_heads * c.head_dim * 4; break;
    case 3: src = h->g; n = B * c.intermediate * 4; break;
    case 4: src = h->sumsq; n = B * (c.hidden / kResGroup) * 4; break;
    default:
      set_err("dec_debug_buffer: unknown buffer %d", which);
      return DEC_ERR_INVALID_ARG;
  }
  if (bytes < n) {
    set_err("dec_debug_buffer: %zu bytes needed", n);
    return DEC_ERR_INVALID_ARG;
  }
  DEC_CUDA(cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)));
  return DEC_OK;
}

extern "C" dec_status dec_set_timeline(dec_handle* h, unsigned long long* stamps) {
  if (!h) {
    set_err("handle is NULL");
    return DEC_ERR_INVALID_ARG;
  }
#if !(defined(DEC_TIMELINE) && DEC_TIMELINE)
  if (stamps) {
    set_err("timeline stamps are compiled in only when the library is built with DEC_TIMELINE=1");
    return DEC_ERR_UNSUPPORTED;
  }
#endif
  h->timeline = stamps;
  drop_graph(h);  // the next step captures the kernels with the new pointer
  return DEC_OK;
}

// ---------------------------------------------------------------- sampling

extern "C" dec_status dec_sample(const float* logits, int batch, int vocab, const dec_sampling_params* params,
                                 int32_t* tokens, dec_stream_t stream) {
  if (!logits || !tokens || !params || batch < 1 || vocab < 1) {
    set_err("dec_sample: NULL logits/tokens/params or batch/vocab < 1");
    return DEC_ERR_INVALID_ARG;
  }
  if (!(params->top_p > 0.f && params->top_p <= 1.f) || !std::isfinite(params->temperature)) {
    set_err("dec_sample: top_p must be in (0, 1] and temperature finite");
    return DEC_ERR_INVALID_ARG;
  }
  SampleParams sp{};
  sp.logits = logits;
  sp.V = vocab;
  sp.temperature = params->temperature;
  sp.top_k = params->top_k;
  sp.top_p = params->top_p;
  sp.seed = params->seed;
  sp.offset = params->offset;
  sp.offset_dev = params->offset_device;
  sp.tokens = tokens;
  DEC_CUDA(launch_sample(reinterpret_cast<cudaStream_t>(stream), sp, batch));
  return DEC_OK;
}

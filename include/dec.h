/*
 * dec.h - C ABI of the GB300 one-token decode step for a Qwen3-style dense decoder.
 *
 * One call of dec_step() runs one greedy decode step for B independent
 * sequences, entirely on the GPU (sm_103a):
 *
 *   h = embed[token]                                   (gather)
 *   for each layer:
 *     xn = RMSNorm(h) * in_norm                        (fused into the QKV GEMV)
 *     q, k, v = Wq xn, Wk xn, Wv xn                    (one fused GEMV)
 *     q, k = per-head RMSNorm (q_norm / k_norm), then rotate-half RoPE at P
 *     cache[P] = bf16(k), bf16(v) (or their affine 8-bit form);
 *     o = softmax(q K^T / sqrt(d)) V over 0..P
 *                                                      (one fused attention kernel,
 *                                                       split over the positions,
 *                                                       log-sum-exp merge)
 *     h += Wo o                                        (GEMV + residual)
 *     h += Wdown(silu(Wgate xn) * (Wup xn)), xn = RMSNorm(h) * post_norm
 *   logits = Wlm RMSNorm(h) * final_norm; argmax      (vocab-tiled GEMV, two-stage argmax)
 *
 * Sources (page title and section):
 *   - ANEForge, "LLMs on the ANE", "What's inside": pre-norm block order,
 *     rotate-half RoPE, GQA (KV heads shared by groups of query heads);
 *     "Correctness": separate head_dim, per-head q/k RMSNorm before RoPE;
 *     "lm_head on the ANE": lm_head tiled along the vocab, greedy argmax.
 *   - Butter, architecture.md, figure "SINGLE-TOKEN DECODE": the kernel
 *     sequence, KV append into a preallocated buffer at offset = cache length,
 *     one command buffer per token (here: one CUDA graph per step); GPU
 *     sampling (greedy argmax on the device, 4-byte result).
 *   - oxinfer crate page, "MLX checkpoints": affine 4-bit weights, eight per
 *     uint32, one bf16 scale and bias per group of 64, w = scale*q + bias.
 *   - Butter, architecture.md, model-layer section (per-layer cache types: KVCache,
 *     AffineQuantizedKVCache): the KV cache may hold affine 8-bit codes (the same
 *     affine form, one bf16 scale and bias per 64 values of a row) instead of bf16.
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device memory of the current device.  Host
 *     pointers (config, weight tables, outputs of size queries) are plain
 *     host memory, read only during the call.
 *   - Functions returning dec_status report host-detectable errors
 *     immediately; the message is available from dec_last_error() (thread
 *     local, valid until the next failing call on the same thread).
 *   - Work is enqueued on the caller's stream and is asynchronous.  CUDA
 *     faults surface at the caller's next synchronisation, or as
 *     DEC_ERR_CUDA from a later call.
 */
#ifndef TOKEN_DECODE_STEP_DEC_H
#define TOKEN_DECODE_STEP_DEC_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DEC_API __attribute__((visibility("default")))
#else
#define DEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (an opaque CUDA stream handle); NULL = legacy default stream. */
typedef struct CUstream_st *dec_stream_t;

typedef enum {
    DEC_OK = 0,
    DEC_ERR_INVALID_ARG = 1,   /* NULL/inconsistent argument */
    DEC_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels handle (see dec_config) */
    DEC_ERR_OOM = 3,           /* cudaMalloc failed */
    DEC_ERR_CUDA = 4,          /* a CUDA runtime call failed */
    DEC_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up (status word bit) */
    DEC_ERR_DEVICE_INPUT = 6   /* a token id or position was out of range (status word bit) */
} dec_status;

typedef enum {
    DEC_W_BF16 = 0,            /* bf16 [out][in] row-major */
    DEC_W_AFFINE4_G64 = 1      /* w = uint32 [out][in/8] (nibble k of word j is input 8j+k,
                                  bits 4k..4k+3), scales, biases = bf16 [out][in/64] */
} dec_wfmt;

typedef enum {
    DEC_KV_BF16 = 0,           /* bf16 [n_layers][2][batch][n_kv_heads][max_ctx][head_dim] */
    DEC_KV_AFFINE8_G64 = 1     /* affine 8-bit, see dec_kv_cache_bytes() for the layout */
} dec_kvfmt;

/* Model and run shape.  Supported (else DEC_ERR_UNSUPPORTED): head_dim in {64, 128};
   n_q_heads / n_kv_heads in {1, 2, 4}; hidden and intermediate multiples of 64;
   vocab >= 1; rows = batch * tokens_per_seq at most 65535 (one row runs CUDA-core GEMV
   kernels, more rows tensor-core kernels, in blocks of 16 rows for bf16 weights and 32
   for affine 4-bit); tokens_per_seq 0..4096 (0 means 1); max_ctx >= 1, and a multiple
   of 16 for the affine 8-bit cache.  Required (else DEC_ERR_INVALID_ARG): every size positive, rms_eps > 0,
   rope_theta > 1, n_q_heads a multiple of n_kv_heads, kv_fmt a dec_kvfmt.

   tokens_per_seq T > 1 makes dec_step a multi-token verify step (speculative decoding's
   check of drafted tokens in one forward: ANEForge "LLMs on the ANE", "Speculative
   decoding"; Butter architecture.md, phase 8): row r = b T + t carries token_ids[r] at position
   positions[b] + t of sequence b, attends causally to that sequence's slots 0 ..
   positions[b] + t, and its K/V are written at that slot; logits_out and argmax_out
   hold one row per (b, t).  The result of row (b, t) is that of a one-token step of
   sequence b at position positions[b] + t after the rows (b, 0..t-1).  The same step with
   T prompt tokens per sequence is a chunked prefill (the step before decode): it fills
   slots positions[b] .. positions[b] + T - 1 with the prompt's K/V in one forward, and the
   last row of each sequence gives the first generated token; logits_out may be NULL. */
/* Kernel family of the projections of steps with 2..32 rows on models of hidden >= 2048 (a
   batch of sequences, or the rows of a verify step).  Both compute the same products.
   TCGEN05 selects the tensor-memory kernels for every projection (bf16 weights streamed by TMA
   into tcgen05.mma; 4-bit codes expanded into tensor memory with a per-group accumulator
   readout), MMA_SYNC the mma.sync kernels over fragment-packed weight tiles.  AUTO takes, per
   projection, what measured faster on this part (8B shapes at 32 rows of 4-bit weights and 8
   rows of bf16): with 4-bit weights and 16 or more rows the gate/up and lm_head projections on
   tcgen05 and the others on mma.sync; with bf16 weights, or fewer rows, mma.sync. */
typedef enum {
    DEC_PROJ_AUTO = 0,
    DEC_PROJ_MMA_SYNC = 1,
    DEC_PROJ_TCGEN05 = 2
} dec_projk;

typedef struct {
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, intermediate, vocab;
    float rms_eps, rope_theta;
    int linear_fmt;            /* dec_wfmt, applies to every linear including lm_head */
    int batch, max_ctx;        /* sequences per step; cache slots per sequence */
    int tokens_per_seq;        /* new tokens per sequence and step: 1 (decode), 2..8 (verify), up to
                                  4096 (a prefill chunk); 0 = 1 */
    int kv_fmt;                /* dec_kvfmt of the KV cache (0 = bf16) */
    int proj_kernels;          /* dec_projk (0 = AUTO); DEC_ERR_INVALID_ARG outside 0..2 */
} dec_config;

/* One linear layer, row-major [out][in] in device memory.  bf16: w only (scales,
   biases ignored).  affine 4-bit: all three, layouts as in dec_wfmt. */
typedef struct {
    const void *w;
    const void *scales;
    const void *biases;
} dec_linear;

typedef struct {
    const void *in_norm;       /* bf16 [hidden] */
    const void *post_norm;     /* bf16 [hidden] */
    const void *q_norm;        /* bf16 [head_dim], shared by the layer's query heads */
    const void *k_norm;        /* bf16 [head_dim], shared by the layer's KV heads */
    dec_linear q, k, v;        /* [n_q*d][hidden], [n_kv*d][hidden], [n_kv*d][hidden] */
    dec_linear o;              /* [hidden][n_q*d] */
    dec_linear gate, up;       /* [intermediate][hidden] */
    dec_linear down;           /* [hidden][intermediate] */
} dec_layer_weights;

typedef struct {
    const void *embed;         /* bf16 [vocab][hidden] (bf16 in every format) */
    const void *final_norm;    /* bf16 [hidden] */
    dec_linear lm_head;        /* [vocab][hidden], untied from embed */
    const dec_layer_weights *layers;   /* host array of n_layers entries */
} dec_weights;

typedef struct dec_handle dec_handle;

/* Validate cfg, allocate the handle's device memory, repack every weight into
   the handle's own layout (device-to-device, on an internal stream that is
   synchronised before returning), and upload the RoPE frequency table.
   (Butter architecture.md, dispatch-mode section: weight buffers are immutable after
   load and bound once, the per-token state stays small; oxinfer crate page, "MLX
   checkpoints": the affine 4-bit layout the packing reads.)  The
   caller may free its weight buffers once this returns.  Returns NULL on
   failure (see dec_last_error()).  Uses the current CUDA device. */
DEC_API dec_handle *dec_create(const dec_config *cfg, const dec_weights *weights);

/* One decode step (Butter "SINGLE-TOKEN DECODE" sequence), enqueued on `stream`.
   With T = tokens_per_seq (1 unless set), rows = batch * T:
     token_ids  device int32 [rows]: input token per row (row b T + t: token t of
                sequence b).
     positions  device int32 [batch]: P_b = cached positions of sequence b; row
                (b, t) writes K/V slot P_b + t, attends over slots 0..P_b + t and
                applies RoPE at angle P_b + t.  The caller advances positions.
     kv_cache   device, dec_kv_cache_bytes(cfg) bytes in the cfg's kv_fmt (layouts at
                dec_kv_cache_bytes), caller-owned, 16-byte aligned.  New K/V rows
                are rounded to bf16, or quantized as dec_kv_quantize() does.
     logits_out device float [rows][vocab], or NULL to skip writing logits.
     argmax_out device int32 [rows]: greedy token (lowest index on equal
                logits).  May alias token_ids (read happens first).
   Out-of-range token ids or positions are clamped on the device and flagged in
   the status word (dec_get_device_status); nothing outside the buffers is
   touched.  By default the step runs as one CUDA graph, re-captured whenever
   the set of pointers changes.  One handle must not be used by two streams at once. */
DEC_API dec_status dec_step(dec_handle *h, const int32_t *token_ids, const int32_t *positions,
                    void *kv_cache, float *logits_out, int32_t *argmax_out,
                    dec_stream_t stream);

/* dec_step for a host-driven decode loop: the token ids, positions and greedy result live
   in host memory (Butter architecture.md, "SINGLE-TOKEN DECODE": one submission per token,
   a 4-byte result read back per sequence).
     token_ids  host int32 [rows], positions host int32 [batch], argmax_out host int32 [rows]
                (may alias token_ids); pageable or pinned.
     kv_cache, logits_out  device, as in dec_step.
   The inputs are copied into the handle's pinned staging buffer; then one CUDA graph on
   `stream` copies them to the device, runs the step and copies the argmax back, and the
   call returns after synchronising `stream` with argmax_out written.  The staging buffers
   (pinned host and device, 4 (2 rows + batch) bytes each) are allocated by the first call
   (DEC_ERR_OOM if that fails) and freed by dec_destroy.  Errors as dec_step; a CUDA fault of
   the step surfaces here as DEC_ERR_CUDA.  The same graph rule as dec_step (re-captured when
   kv_cache or logits_out changes); the two calls keep separate graphs. */
DEC_API dec_status dec_step_host(dec_handle *h, const int32_t *token_ids, const int32_t *positions,
                    void *kv_cache, float *logits_out, int32_t *argmax_out,
                    dec_stream_t stream);

/* Free every device resource of the handle (caller buffers are untouched).
   The caller must make sure no step of this handle is still running.  (The end of
   the load-time binding of Butter architecture.md, dispatch-mode section: what
   dec_create bound once is released once.) */
DEC_API void dec_destroy(dec_handle *h);

/* Bytes of the KV cache for cfg (0 if cfg is NULL or invalid): the caller preallocates the
   whole cache once and each step appends at offset = cache length (Butter architecture.md,
   figure "SINGLE-TOKEN DECODE", cache.append; ANEForge "LLMs on the ANE", "Prefill and
   decode": a resident KV cache).  Plane 0 holds the keys (after the per-head norm and
   RoPE), plane 1 the values; slot s of a sequence holds its position s.
     DEC_KV_BF16: bf16 [n_layers][2][batch][n_kv_heads][max_ctx][head_dim].
     DEC_KV_AFFINE8_G64: the codes, uint8 [n_layers][2][batch][n_kv_heads][max_ctx][head_dim],
       then, from the first multiple of 256 bytes after them, the (scale, bias) pairs, bf16
       [n_layers][2][batch][n_kv_heads][max_ctx][head_dim/64][2]: element i of a row reads
       scale[i/64] * code[i] + bias[i/64]. */
DEC_API size_t dec_kv_cache_bytes(const dec_config *cfg);

/* Test hook: the tensor-core projection kernel of long prefill chunks (tcgen05.mma with TMA
   operands, the accumulator in tensor memory) on caller buffers, plain store epilogue:
   out[m][n] = sum_k (x_hi[m][k] + x_lo[m][k]) * w[n][k] in fp32.
     x_hl  device bf16 [2][M][K] (plane 0 hi, plane 1 lo), 16-byte aligned
     w     device bf16 [N][K] row-major, 16-byte aligned
     out   device float [M][N]
   persistent: 0 = one CTA per tile; 1 = the persistent form (one CTA per SM walking the tiles,
   TMA / MMA / epilogue warps, two accumulators so that an epilogue overlaps the next tile's
   MMAs), the one dec_step uses.
   K a positive multiple of 64, M and N >= 1 (else DEC_ERR_INVALID_ARG).  One launch on `stream`. */
DEC_API dec_status dec_debug_gemm_tc5(const void *x_hl, int M, const void *w, int N, int K, float *out,
                                      int persistent, dec_stream_t stream);

/* Test hook for the time-out path: enqueues on `stream` one bounded wait that can only run out
   (an mbarrier that nothing arrives on, polled `polls` times, 1..65536), which sets the
   time-out bit of h's device status word exactly as a bounded wait of the tensor-memory kernels
   does when a copy or an MMA never completes.  After a stream synchronisation,
   dec_get_device_status returns DEC_ERR_TIMEOUT (and clears the word); the handle and the CUDA
   context stay usable.  No GPU fault or trap is involved. */
DEC_API dec_status dec_debug_force_timeout(dec_handle *h, int polls, dec_stream_t stream);

/* Test hook: the tensor-core projection kernel of batched decode steps with affine 4-bit weights
   (oxinfer crate page, "MLX checkpoints": w = scale * q + bias per group of 64, so that
   sum_k w_k x_k = scale * sum_k (128 + q_k) x_k + (bias - 128 scale) * sum_k x_k): the codes are
   expanded exactly to bf16 (128 + q) into tensor memory, tcgen05.mma forms each group's sum (and,
   through rows of ones, the sum of x) into tensor memory, and the scale and bias are applied per
   group in float32; on caller buffers, plain store epilogue:
     out[m][n] = sum_k (x_hi[m][k] + x_lo[m][k]) * w[n][k],  w = fl(scale * q + bias) per group of 64.
     x_hl      device bf16 [2][M][K] (plane 0 hi, plane 1 lo), 16-byte aligned, M in 1..32
     codes     device uint32 [N][K/8] (element 8 j + k in bits 4k..4k+3 of word j), 16-byte aligned
     sb        device uint32 [N][K/64]: bf16 scale bits | bf16 bias bits << 16, 16-byte aligned
     out       device float [M][N]
     S         K splits (dividing K / 64); S > 1 needs partials (device float [S][M][N]) and
               counters (device uint32 [ceil(N / 120) + 1]: one per 120-row tile, zero, left zero)
   K a positive multiple of 64, N >= 1 (else DEC_ERR_INVALID_ARG).  One launch on `stream`. */
DEC_API dec_status dec_debug_gemm_q4tc(const void *x_hl, int M, const void *codes, const void *sb, int N, int K,
                    int S, float *out, float *partials, unsigned *counters, dec_stream_t stream);

/* Test hook: the bf16 form of the batched-decode tensor-core projection (weights streamed by TMA
   into the MMA, stream-K schedule) on caller buffers, plain store:
   out[m][n] = sum_k (x_hi[m][k] + x_lo[m][k]) w[n][k].
     x_hl      device bf16 [2][M][K], 16-byte aligned, M in 1..32
     w         device bf16 [N][K] row-major, 16-byte aligned
     out       device float [M][N]
     ctas      CTAs of the schedule (<= 0: one per SM); the tiles' 64-input stages are dealt to
               them in contiguous ranges
     partials  device float [K/64][M][N] (slots for the segments of a tile shared by CTAs)
     counters  device uint32 [ceil(N / 128) + 1], zero, left zero
   K a positive multiple of 64, N >= 1 (else DEC_ERR_INVALID_ARG).  One launch on `stream`. */
DEC_API dec_status dec_debug_gemm_btc(const void *x_hl, int M, const void *w, int N, int K, int ctas, float *out,
                    float *partials, unsigned *counters, dec_stream_t stream);

/* Test hook (host only, no CUDA call): the partial-result slots that the stream-K schedule of
   dec_debug_gemm_btc needs for an N x K projection on `ctas` CTAs, i.e. the most CTAs that
   share one 128-row tile; 0 for a non-positive argument. */
DEC_API int dec_debug_btc_max_segments(int N, int K, int ctas);

/* Test hook (host only, no CUDA call): the kernel family that each projection of a handle
   created from *cfg runs on, as dec_config.proj_kernels selects it (the projection kernel
   family, above).  Bit i of *tcgen05_mask is set when projection i (0 q/k/v, 1 o, 2 gate/up,
   3 down, 4 lm_head) runs on a tcgen05 decode kernel (k_gemm_q4tc for 4-bit weights,
   k_gemm_btc for bf16) rather than the mma.sync kernel, the batch-1 GEMV or the prefill GEMM.
     cfg           host pointer; the config dec_create would check (same checks, same status)
     tcgen05_mask  host int, written on success
   DEC_ERR_INVALID_ARG for a NULL argument; a config that dec_create refuses gets its status. */
DEC_API dec_status dec_debug_proj_plan(const dec_config *cfg, int *tcgen05_mask);

/* The affine 8-bit quantizer of the KV cache (the one dec_step applies to new rows), on
   caller buffers.  For each group of 64 consecutive values x of a row, in float32:
   mn, mx = min, max; scale = bf16(fl(fl(mx - mn) / 255)); bias = bf16(mn) (round to
   nearest even); code = clamp(rint(fl(fl(x - bias) / scale)), 0, 255), rint rounding
   halves to even, code 0 where scale = 0.  (Butter architecture.md, model-layer section:
   AffineQuantizedKVCache; the affine form of oxinfer's "MLX checkpoints" section.)
     src     device float [rows][head_dim], finite values
     codes   device uint8 [rows][head_dim]
     params  device bf16 [rows][head_dim/64][2]: (scale, bias) per group
   head_dim 64 or 128 (else DEC_ERR_UNSUPPORTED); rows >= 0; NULL pointers with rows > 0
   -> DEC_ERR_INVALID_ARG.  One kernel launch on `stream`. */
DEC_API dec_status dec_kv_quantize(const float *src, int rows, int head_dim, uint8_t *codes, void *params,
                                   dec_stream_t stream);

/* Message of the last failing call on this thread ("" if none).  (The error side of a C
   API over the engine, as the oxinfer crate page lists one, capi feature and
   include/oxinfer.h; the page gives no error convention, so this one is a plain
   status code plus a thread-local message.) */
DEC_API const char *dec_last_error(void);

/* Read and clear the device status word (call after synchronising the stream of
   the steps in question).  The step never reads the token ids or positions back to the
   host (Butter architecture.md, GPU sampling section: the greedy token stays on the
   device, a 4-byte result), so range errors the kernels detect are recorded here.  *out receives the raw bits (1: token id out of range,
   2: position out of range, 4: bounded wait timed out).  Returns DEC_OK when the
   word was 0, DEC_ERR_DEVICE_INPUT / DEC_ERR_TIMEOUT otherwise. */
DEC_API dec_status dec_get_device_status(dec_handle *h, int *out);

/* Test hook (oxinfer crate page, "MLX checkpoints": w = scale * q + bias per group of
   64, eight codes per uint32): write the dequantised weights of one linear as float32
   [out][in] (row-major, canonical row order) to device memory `out`, computed from the
   handle's packed copy with the same nibble unpacking the GEMV kernels use and a
   single rounding (fmaf(scale, q, bias)); for bf16 the exact value.
   which: 0 q, 1 k, 2 v, 3 o, 4 gate, 5 up, 6 down, 7 lm_head (layer ignored). */
DEC_API dec_status dec_debug_dequant(dec_handle *h, int layer, int which, float *out, dec_stream_t stream);

/* Greedy feedback helper: token_ids[b] = argmax[b]; positions[b] += 1, for b < batch,
   as one small kernel on `stream` (device pointers). */
DEC_API dec_status dec_advance(const int32_t *argmax, int32_t *token_ids, int32_t *positions, int batch,
                       dec_stream_t stream);

/* 1 (default): dec_step replays a captured CUDA graph; 0: launch kernels one by one. */
DEC_API dec_status dec_set_graph_mode(dec_handle *h, int enabled);

/* Kernel classes reported by dec_profile_step. */
enum {
    DEC_K_EMBED = 0, DEC_K_QKV = 1, DEC_K_ATTN = 2, DEC_K_OPROJ = 3, DEC_K_GATEUP = 4,
    DEC_K_DOWN = 5, DEC_K_LMHEAD = 6, DEC_K_COUNT = 7
};

/* Run one step with individual launches, one after another, each bracketed by CUDA
   events recorded on `stream` (the stream is first held by a short sleeping kernel on
   an internal stream, so that every launch is enqueued before the first runs and the
   times hold no host launch gaps), then synchronise `stream` and add each launch's
   elapsed time (ms) to ms[class] and 1 to launches[class] (host arrays of
   n_classes >= DEC_K_COUNT entries).  Same arguments and results as dec_step. */
DEC_API dec_status dec_profile_step(dec_handle *h, const int32_t *token_ids, const int32_t *positions,
                            void *kv_cache, float *logits_out, int32_t *argmax_out,
                            dec_stream_t stream, double *ms, int *launches, int n_classes);

/* Algorithmic bytes one launch of a kernel class moves at cached length P (same P
   for all sequences): weights (+ norms) read once, KV rows 0..P read, activations
   excluded.  Host-side arithmetic on the handle's config. */
DEC_API double dec_kernel_bytes(const dec_handle *h, int kernel_class, double mean_cached_len);

/* Number of kernels one dec_step launches: 2 + 5 n_layers, or 2 + 6 n_layers for a
   verify step (tokens_per_seq > 1: a K/V append kernel precedes each attention). */
DEC_API int dec_launches_per_step(const dec_handle *h);

/* Kernel-level entry point: the fused attention that dec_step runs for each layer
   (per-head q/k RMSNorm, rotate-half RoPE at positions[b], append of k, v (in the cache format) at
   slot positions[b] of `layer`, split-KV GQA attention over slots 0..positions[b]
   with a log-sum-exp merge), on caller buffers.  ANEForge "LLMs on the ANE",
   "Correctness" and "What's inside"; Butter architecture.md "SINGLE-TOKEN DECODE"
   (rope, cache.append, sdpa_decode).
     cfg        uses n_layers, batch, n_q_heads, n_kv_heads, head_dim, max_ctx,
                rms_eps, rope_theta (same limits as dec_create; any batch >= 1);
                tokens_per_seq must be 0 or 1.
     qkv        device float [batch][(n_q + 2 n_kv) * head_dim]: the new token's raw
                projections, q heads, then k heads, then v heads, head j at j*head_dim.
     q_norm, k_norm  device bf16 [head_dim].
     positions  device int32 [batch], as in dec_step (clamped if out of range).
     kv_cache   as in dec_step (either kv_fmt); only slot positions[b] of `layer` is
                written.
     out        device float [batch][n_q * head_dim]: attention output per query head.
     workspace  caller-owned device scratch (the RoPE table) of at least
                dec_attention_workspace_bytes(cfg) bytes, 256-byte aligned; its
                contents on entry do not matter; one call at a time per workspace.
   Enqueued on `stream`. */
DEC_API size_t dec_attention_workspace_bytes(const dec_config *cfg);
DEC_API dec_status dec_attention(const dec_config *cfg, int layer, const float *qkv, const void *q_norm,
                                 const void *k_norm, const int32_t *positions, void *kv_cache, float *out,
                                 void *workspace, size_t workspace_bytes, dec_stream_t stream);

/* Test hooks for kernel-by-kernel parity.  dec_debug_step_prefix runs the first
   n_launches kernels of one step (embedding = launch 1, then per layer QKV,
   (K/V append for a verify step,) attention, O, gate/up, down, finally lm_head) as
   individual launches.  dec_debug_buffer copies a workspace buffer of the handle to
   device memory dst (rows = batch * tokens_per_seq):
   which 0: residual h float [rows][hidden]; 1: q,k,v projections float
   [rows][(n_q + 2 n_kv) head_dim]; 2: attention output float [rows][n_q head_dim];
   3: SwiGLU output float [rows][intermediate]; 4: residual sums of squares float
   [rows][hidden / 8].  Both enqueue on `stream`. */
DEC_API dec_status dec_debug_step_prefix(dec_handle *h, const int32_t *token_ids, const int32_t *positions,
                                         void *kv_cache, float *logits_out, int32_t *argmax_out,
                                         dec_stream_t stream, int n_launches);
DEC_API dec_status dec_debug_buffer(dec_handle *h, int which, void *dst, size_t bytes, dec_stream_t stream);

/* Test hook: with stamps != NULL, every kernel of later steps records %globaltimer
   values (nanoseconds) in stamps[3 i + 0..2] for launch i of the step (same order
   as dec_debug_step_prefix): 0 = first CTA started (atomic min), 1 = first CTA past
   its wait for the previous kernel (min), 2 = last CTA finished (max).  The caller
   owns the device buffer (3 * dec_launches_per_step() entries) and resets it to
   (~0, ~0, 0) triples before a step.  NULL turns the stamps off.  The step graph
   is re-captured on the next dec_step.  The stamps exist only in a library built
   with DEC_TIMELINE=1 (they cost the GEMV kernels registers); elsewhere a non-NULL
   `stamps` returns DEC_ERR_UNSUPPORTED. */
DEC_API dec_status dec_set_timeline(dec_handle *h, unsigned long long *stamps);

/* dec_attention without a workspace: same arguments, same computation and same
   result as dec_attention, but it allocates nothing and takes no scratch from the
   caller.  The pages have no counterpart; it exists for callers that cannot call
   cudaMalloc at this point -- for example code running while a stream is being
   captured into a CUDA graph in global capture mode (where cudaMalloc is not
   allowed), plug-in or real-time hosts that hand over only input and output
   buffers and forbid device allocations (cudaMalloc can synchronise the device and
   can fail under memory pressure), or hosts whose allocator owns all free memory.
   Its scratch -- the RoPE (cos, sin) table that its first kernel writes and the
   attention kernel reads -- is one fixed array of 1 MiB inside this library;
   every GPU that loads the library holds that array until the process exits.
   Batches whose table exceeds it (more than 2048 sequences at head_dim 128, 4096
   at head_dim 64) are rejected with DEC_ERR_UNSUPPORTED and a message.
     - The first call on each device does a one-time set-up (it looks up the
       array's device address and sets the kernels' shared-memory limit) with that
       device current; make that first call before any stream capture.
     - Every call shares the one array and it keeps the last call's contents;
       each call rewrites the whole table before reading it, so nothing has to
       start at zero.  Calls whose work overlaps on the GPU (other streams, other
       host threads) race on the array; serialise them.
   Enqueued on `stream` (a RoPE-table kernel, then the attention kernel). */
DEC_API dec_status dec_attention_noalloc(const dec_config *cfg, int layer, const float *qkv, const void *q_norm,
                                         const void *k_norm, const int32_t *positions, void *kv_cache, float *out,
                                         dec_stream_t stream);

/* ---- On-device sampling (Butter architecture.md, GPU sampling section: the sampling
   kernel after the lm_head; temperature, top-k, top-p, inverse-CDF draw, 4-byte
   token out).  Per row b of logits [batch][vocab] (float32, device):
     temperature <= 0: tokens[b] = argmax (lowest index on ties);
     else: the k most likely tokens, k = top_k if 1 <= top_k <= 1024, else 1024 (at
     most vocab), ordered by (logit descending, index ascending); p_j = exp((l_j -
     l_0) / temperature); if top_p < 1, the shortest prefix whose cumulative p reaches
     top_p times the sum; tokens[b] = the first kept candidate whose cumulative p
     exceeds u times the kept sum, where u = (x0 >> 8) * 2^-24 and x0 is the first
     word of Philox4x32-10 with key (seed low, seed high 32 bits) and counter (offset
     low, offset high, b, 0).  When offset_device is not NULL the offset is read from
     that device word when the kernel runs (so a captured graph can advance it).
   Logits of -0 rank as +0 and NaN below every number.  One kernel launch on
   `stream`, no allocation.  Errors: NULL logits/tokens/params, batch or vocab < 1,
   top_p not in (0, 1] or a non-finite temperature -> DEC_ERR_INVALID_ARG. */
typedef struct dec_sampling_params {
    float temperature;
    int top_k;
    float top_p;
    unsigned long long seed;
    unsigned long long offset;
    const unsigned long long *offset_device;
} dec_sampling_params;

DEC_API dec_status dec_sample(const float *logits, int batch, int vocab, const dec_sampling_params *params,
                              int32_t *tokens, dec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TOKEN_DECODE_STEP_DEC_H */

"""ctypes binding of include/dec.h (argument marshalling only).

Every function here forwards to the C ABI of ``libdec.so``; all computation of
the decode step runs in that library's CUDA kernels.  The library must have
been built (``token_decode_step_gb300.build.build()``); importing this module
without it raises, there is no fallback path.
"""

from __future__ import annotations

import ctypes
import pathlib

_LIB_PATH = pathlib.Path(__file__).resolve().parent / "libdec.so"

DEC_OK = 0
DEC_ERR_INVALID_ARG = 1
DEC_ERR_UNSUPPORTED = 2
DEC_ERR_OOM = 3
DEC_ERR_CUDA = 4
DEC_ERR_TIMEOUT = 5
DEC_ERR_DEVICE_INPUT = 6

DEC_W_BF16 = 0
DEC_W_AFFINE4_G64 = 1

DEC_KV_BF16 = 0
DEC_KV_AFFINE8_G64 = 1

DEC_PROJ_AUTO = 0
DEC_PROJ_MMA_SYNC = 1
DEC_PROJ_TCGEN05 = 2

DEC_K_EMBED, DEC_K_QKV, DEC_K_ATTN, DEC_K_OPROJ, DEC_K_GATEUP, DEC_K_DOWN, DEC_K_LMHEAD, DEC_K_COUNT = range(8)
KERNEL_CLASS_NAMES = ["embed", "qkv", "attention", "o_proj", "gate_up", "down", "lm_head"]


class SamplingParams(ctypes.Structure):
    """dec_sampling_params (include/dec.h)."""
    _fields_ = [
        ("temperature", ctypes.c_float), ("top_k", ctypes.c_int), ("top_p", ctypes.c_float),
        ("seed", ctypes.c_ulonglong), ("offset", ctypes.c_ulonglong), ("offset_device", ctypes.c_void_p),
    ]


class DecConfig(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_q_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("intermediate", ctypes.c_int),
        ("vocab", ctypes.c_int), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("linear_fmt", ctypes.c_int), ("batch", ctypes.c_int), ("max_ctx", ctypes.c_int),
        ("tokens_per_seq", ctypes.c_int), ("kv_fmt", ctypes.c_int), ("proj_kernels", ctypes.c_int),
    ]


class DecLinear(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p)]


class DecLayerWeights(ctypes.Structure):
    _fields_ = [
        ("in_norm", ctypes.c_void_p), ("post_norm", ctypes.c_void_p), ("q_norm", ctypes.c_void_p),
        ("k_norm", ctypes.c_void_p), ("q", DecLinear), ("k", DecLinear), ("v", DecLinear),
        ("o", DecLinear), ("gate", DecLinear), ("up", DecLinear), ("down", DecLinear),
    ]


class DecWeights(ctypes.Structure):
    _fields_ = [
        ("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p), ("lm_head", DecLinear),
        ("layers", ctypes.POINTER(DecLayerWeights)),
    ]


def _load() -> ctypes.CDLL:
    if not _LIB_PATH.exists():
        raise ImportError(f"{_LIB_PATH} is missing: build it with token_decode_step_gb300.build.build()")
    lib = ctypes.CDLL(str(_LIB_PATH))
    vp, i32p = ctypes.c_void_p, ctypes.c_void_p
    sig = {
        "dec_create": (vp, [ctypes.POINTER(DecConfig), ctypes.POINTER(DecWeights)]),
        "dec_step": (ctypes.c_int, [vp, i32p, i32p, vp, vp, i32p, vp]),
        "dec_step_host": (ctypes.c_int, [vp, i32p, i32p, vp, vp, i32p, vp]),
        "dec_destroy": (None, [vp]),
        "dec_kv_cache_bytes": (ctypes.c_size_t, [ctypes.POINTER(DecConfig)]),
        "dec_last_error": (ctypes.c_char_p, []),
        "dec_get_device_status": (ctypes.c_int, [vp, ctypes.POINTER(ctypes.c_int)]),
        "dec_debug_dequant": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, vp]),
        "dec_advance": (ctypes.c_int, [i32p, i32p, i32p, ctypes.c_int, vp]),
        "dec_set_graph_mode": (ctypes.c_int, [vp, ctypes.c_int]),
        "dec_profile_step": (ctypes.c_int, [vp, i32p, i32p, vp, vp, i32p, vp,
                                            ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int),
                                            ctypes.c_int]),
        "dec_kernel_bytes": (ctypes.c_double, [vp, ctypes.c_int, ctypes.c_double]),
        "dec_launches_per_step": (ctypes.c_int, [vp]),
        "dec_debug_step_prefix": (ctypes.c_int, [vp, i32p, i32p, vp, vp, i32p, vp, ctypes.c_int]),
        "dec_debug_buffer": (ctypes.c_int, [vp, ctypes.c_int, vp, ctypes.c_size_t, vp]),
        "dec_set_timeline": (ctypes.c_int, [vp, vp]),
        "dec_attention_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(DecConfig)]),
        "dec_attention": (ctypes.c_int, [ctypes.POINTER(DecConfig), ctypes.c_int, vp, vp, vp, vp, vp, vp, vp,
                                         ctypes.c_size_t, vp]),
        "dec_attention_noalloc": (ctypes.c_int, [ctypes.POINTER(DecConfig), ctypes.c_int, vp, vp, vp, vp, vp, vp,
                                                 vp]),
        "dec_sample": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(SamplingParams), vp, vp]),
        "dec_kv_quantize": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, vp, vp]),
        "dec_debug_gemm_tc5": (ctypes.c_int, [vp, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp]),
        "dec_debug_force_timeout": (ctypes.c_int, [vp, ctypes.c_int, vp]),
        "dec_debug_gemm_q4tc": (ctypes.c_int, [vp, ctypes.c_int, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp,
                                               vp, vp, vp]),
        "dec_debug_gemm_btc": (ctypes.c_int, [vp, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp,
                                              vp, vp]),
        "dec_debug_btc_max_segments": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
        "dec_debug_proj_plan": (ctypes.c_int, [ctypes.POINTER(DecConfig), ctypes.POINTER(ctypes.c_int)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class DecError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status}: {dec_last_error()}")
        self.status = status


def _check(status: int, where: str) -> int:
    if status != DEC_OK:
        raise DecError(status, where)
    return status


# ------------------------------------------------------------------ the C functions, same names

def dec_last_error() -> str:
    return (lib.dec_last_error() or b"").decode()


def dec_kv_cache_bytes(cfg: DecConfig) -> int:
    return int(lib.dec_kv_cache_bytes(ctypes.byref(cfg)))


def dec_create(cfg: DecConfig, weights: DecWeights) -> int:
    """Returns the handle (an integer address); raises DecError on failure."""
    h = lib.dec_create(ctypes.byref(cfg), ctypes.byref(weights))
    if not h:
        raise DecError(-1, "dec_create")
    return h


def dec_step(h: int, token_ids: int, positions: int, kv_cache: int, logits_out: int | None, argmax_out: int,
             stream: int = 0) -> int:
    return _check(lib.dec_step(h, token_ids, positions, kv_cache, logits_out, argmax_out, stream), "dec_step")


def dec_step_host(h: int, token_ids: int, positions: int, kv_cache: int, logits_out: int | None,
                  argmax_out: int, stream: int = 0) -> int:
    """token_ids, positions and argmax_out are HOST addresses; returns after the step."""
    return _check(lib.dec_step_host(h, token_ids, positions, kv_cache, logits_out, argmax_out, stream),
                  "dec_step_host")


def dec_destroy(h: int) -> None:
    lib.dec_destroy(h)


def dec_get_device_status(h: int) -> tuple[int, int]:
    out = ctypes.c_int(0)
    st = lib.dec_get_device_status(h, ctypes.byref(out))
    return st, out.value


def dec_debug_dequant(h: int, layer: int, which: int, out: int, stream: int = 0) -> int:
    return _check(lib.dec_debug_dequant(h, layer, which, out, stream), "dec_debug_dequant")


def dec_advance(argmax: int, token_ids: int, positions: int, batch: int, stream: int = 0) -> int:
    return _check(lib.dec_advance(argmax, token_ids, positions, batch, stream), "dec_advance")


def dec_set_graph_mode(h: int, enabled: bool) -> int:
    return _check(lib.dec_set_graph_mode(h, 1 if enabled else 0), "dec_set_graph_mode")


def dec_profile_step(h: int, token_ids: int, positions: int, kv_cache: int, logits_out: int | None,
                     argmax_out: int, stream: int, ms: list[float], launches: list[int]) -> None:
    """Adds per-kernel-class milliseconds and launch counts into ``ms`` / ``launches``."""
    cms = (ctypes.c_double * DEC_K_COUNT)(*ms)
    cl = (ctypes.c_int * DEC_K_COUNT)(*launches)
    _check(lib.dec_profile_step(h, token_ids, positions, kv_cache, logits_out, argmax_out, stream, cms, cl,
                                DEC_K_COUNT), "dec_profile_step")
    ms[:] = list(cms)
    launches[:] = list(cl)


def dec_kernel_bytes(h: int, kernel_class: int, mean_cached_len: float) -> float:
    return float(lib.dec_kernel_bytes(h, kernel_class, mean_cached_len))


def dec_launches_per_step(h: int) -> int:
    return int(lib.dec_launches_per_step(h))


def dec_attention_workspace_bytes(cfg: DecConfig) -> int:
    return int(lib.dec_attention_workspace_bytes(ctypes.byref(cfg)))


def dec_attention(cfg: DecConfig, layer: int, qkv: int, q_norm: int, k_norm: int, positions: int, kv_cache: int,
                  out: int, workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    return _check(lib.dec_attention(ctypes.byref(cfg), layer, qkv, q_norm, k_norm, positions, kv_cache, out,
                                    workspace, workspace_bytes, stream), "dec_attention")


def dec_attention_noalloc(cfg: DecConfig, layer: int, qkv: int, q_norm: int, k_norm: int, positions: int,
                          kv_cache: int, out: int, stream: int = 0) -> int:
    return _check(lib.dec_attention_noalloc(ctypes.byref(cfg), layer, qkv, q_norm, k_norm, positions, kv_cache,
                                            out, stream), "dec_attention_noalloc")


def dec_sample(logits: int, batch: int, vocab: int, params: SamplingParams, tokens: int, stream: int = 0) -> int:
    return _check(lib.dec_sample(logits, batch, vocab, ctypes.byref(params), tokens, stream), "dec_sample")


def dec_debug_gemm_tc5(x_hl: int, M: int, w: int, N: int, K: int, out: int, persistent: int = 1,
                       stream: int = 0) -> int:
    return _check(lib.dec_debug_gemm_tc5(x_hl, M, w, N, K, out, persistent, stream), "dec_debug_gemm_tc5")


def dec_debug_force_timeout(h: int, polls: int = 256, stream: int = 0) -> int:
    return _check(lib.dec_debug_force_timeout(h, polls, stream), "dec_debug_force_timeout")


def dec_debug_gemm_q4tc(x_hl: int, M: int, codes: int, sb: int, N: int, K: int, S: int, out: int,
                        partials: int | None = None, counters: int | None = None, stream: int = 0) -> int:
    return _check(lib.dec_debug_gemm_q4tc(x_hl, M, codes, sb, N, K, S, out, partials, counters, stream),
                  "dec_debug_gemm_q4tc")


def dec_debug_gemm_btc(x_hl: int, M: int, w: int, N: int, K: int, ctas: int, out: int, partials: int,
                       counters: int, stream: int = 0) -> int:
    return _check(lib.dec_debug_gemm_btc(x_hl, M, w, N, K, ctas, out, partials, counters, stream),
                  "dec_debug_gemm_btc")


def dec_debug_proj_plan(cfg: DecConfig) -> int:
    """Bit mask of the projections (0 q/k/v, 1 o, 2 gate/up, 3 down, 4 lm_head) on tcgen05 kernels."""
    mask = ctypes.c_int(-1)
    _check(lib.dec_debug_proj_plan(ctypes.byref(cfg), ctypes.byref(mask)), "dec_debug_proj_plan")
    return mask.value


def dec_kv_quantize(src: int, rows: int, head_dim: int, codes: int, params: int, stream: int = 0) -> int:
    return _check(lib.dec_kv_quantize(src, rows, head_dim, codes, params, stream), "dec_kv_quantize")


def dec_debug_step_prefix(h: int, token_ids: int, positions: int, kv_cache: int, logits_out: int | None,
                          argmax_out: int, stream: int, n_launches: int) -> int:
    return _check(lib.dec_debug_step_prefix(h, token_ids, positions, kv_cache, logits_out, argmax_out, stream,
                                            n_launches), "dec_debug_step_prefix")


def dec_debug_buffer(h: int, which: int, dst: int, nbytes: int, stream: int = 0) -> int:
    return _check(lib.dec_debug_buffer(h, which, dst, nbytes, stream), "dec_debug_buffer")


def dec_set_timeline(h: int, stamps: int | None) -> int:
    return _check(lib.dec_set_timeline(h, stamps), "dec_set_timeline")

"""Marshalling from PyTorch tensors to the C ABI (device pointers and sizes only).

PyTorch provides device memory and streams here; every step of the decode path
runs in libdec.so's kernels.
"""

from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import dec


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "expected a contiguous CUDA tensor"
    return t.data_ptr()


def make_config(shape, batch: int | None = None, max_ctx: int | None = None,
                tokens_per_seq: int = 1, proj_kernels: int = dec.DEC_PROJ_AUTO) -> dec.DecConfig:
    """dec_config from any object with the model-shape attributes (n_layers, hidden, ...,
    and optionally kv_format "bf16" / "affine8_g64")."""
    fmt = dec.DEC_W_BF16 if shape.weight_format == "bf16" else dec.DEC_W_AFFINE4_G64
    kv_fmt = dec.DEC_KV_AFFINE8_G64 if getattr(shape, "kv_format", "bf16") == "affine8_g64" else dec.DEC_KV_BF16
    return dec.DecConfig(kv_fmt=kv_fmt, proj_kernels=proj_kernels,
                         **_shape_fields(shape, fmt, batch, max_ctx, tokens_per_seq))


def _shape_fields(shape, fmt, batch, max_ctx, tokens_per_seq) -> dict:
    return dict(
        n_layers=shape.n_layers, hidden=shape.hidden, n_q_heads=shape.n_q_heads, n_kv_heads=shape.n_kv_heads,
        head_dim=shape.head_dim, intermediate=shape.intermediate, vocab=shape.vocab, rms_eps=shape.rms_eps,
        rope_theta=shape.rope_theta, linear_fmt=fmt, batch=batch if batch is not None else shape.batch,
        max_ctx=max_ctx if max_ctx is not None else shape.max_ctx, tokens_per_seq=tokens_per_seq)


def kv_quantize(src: torch.Tensor, codes: torch.Tensor, params: torch.Tensor) -> None:
    """dec_kv_quantize on CUDA tensors: src float32 [rows, d], codes uint8 [rows, d], params
    bf16 [rows, d/64, 2]."""
    rows, d = src.shape
    dec.dec_kv_quantize(_ptr(src), rows, d, _ptr(codes), _ptr(params), torch.cuda.current_stream().cuda_stream)


def _linear(x) -> dec.DecLinear:
    if isinstance(x, dict):
        return dec.DecLinear(_ptr(x["w"]), _ptr(x["scales"]), _ptr(x["biases"]))
    return dec.DecLinear(_ptr(x), None, None)


class Decoder:
    """Owns one dec_handle built from a dict of CUDA weight tensors laid out as in
    include/dec.h (embed, final_norm, lm_head, layers[i][in_norm, post_norm, q_norm,
    k_norm, q, k, v, o, gate, up, down])."""

    def __init__(self, shape, weights: dict, batch: int | None = None, max_ctx: int | None = None,
                 tokens_per_seq: int = 1, proj_kernels: int = dec.DEC_PROJ_AUTO):
        self.cfg = make_config(shape, batch, max_ctx, tokens_per_seq, proj_kernels)
        L = self.cfg.n_layers
        layers = (dec.DecLayerWeights * L)()
        for i, lw in enumerate(weights["layers"][:L]):
            layers[i] = dec.DecLayerWeights(
                _ptr(lw["in_norm"]), _ptr(lw["post_norm"]), _ptr(lw["q_norm"]), _ptr(lw["k_norm"]),
                _linear(lw["q"]), _linear(lw["k"]), _linear(lw["v"]), _linear(lw["o"]),
                _linear(lw["gate"]), _linear(lw["up"]), _linear(lw["down"]))
        w = dec.DecWeights(_ptr(weights["embed"]), _ptr(weights["final_norm"]), _linear(weights["lm_head"]),
                           ctypes.cast(layers, ctypes.POINTER(dec.DecLayerWeights)))
        self.handle = dec.dec_create(self.cfg, w)

    @property
    def kv_cache_bytes(self) -> int:
        return dec.dec_kv_cache_bytes(self.cfg)

    def step(self, tokens: torch.Tensor, positions: torch.Tensor, kv: torch.Tensor, logits: torch.Tensor | None,
             argmax: torch.Tensor, stream: torch.cuda.Stream | None = None) -> None:
        s = (stream or torch.cuda.current_stream()).cuda_stream
        dec.dec_step(self.handle, _ptr(tokens), _ptr(positions), _ptr(kv), _ptr(logits), _ptr(argmax), s)

    def step_host(self, tokens: np.ndarray, positions: np.ndarray, kv: torch.Tensor, logits: torch.Tensor | None,
                  argmax: np.ndarray, stream: torch.cuda.Stream | None = None) -> None:
        """One step with host int32 arrays (C-contiguous numpy) for tokens, positions and the argmax."""
        for a in (tokens, positions, argmax):
            if a.dtype != np.int32 or not a.flags["C_CONTIGUOUS"]:
                raise ValueError("tokens, positions and argmax must be C-contiguous int32 numpy arrays")
        rows = self.cfg.batch * max(1, self.cfg.tokens_per_seq)
        if tokens.size < rows or positions.size < self.cfg.batch or argmax.size < rows:
            raise ValueError("host arrays are smaller than the step's rows / batch")
        s = (stream or torch.cuda.current_stream()).cuda_stream
        dec.dec_step_host(self.handle, tokens.ctypes.data, positions.ctypes.data, _ptr(kv), _ptr(logits),
                          argmax.ctypes.data, s)

    def profile_step(self, tokens, positions, kv, logits, argmax, ms: list[float], launches: list[int],
                     stream: torch.cuda.Stream | None = None) -> None:
        s = (stream or torch.cuda.current_stream()).cuda_stream
        dec.dec_profile_step(self.handle, _ptr(tokens), _ptr(positions), _ptr(kv), _ptr(logits), _ptr(argmax),
                             s, ms, launches)

    def advance(self, argmax: torch.Tensor, tokens: torch.Tensor, positions: torch.Tensor,
                stream: torch.cuda.Stream | None = None) -> None:
        s = (stream or torch.cuda.current_stream()).cuda_stream
        dec.dec_advance(_ptr(argmax), _ptr(tokens), _ptr(positions), tokens.numel(), s)

    def set_graph_mode(self, enabled: bool) -> None:
        dec.dec_set_graph_mode(self.handle, enabled)

    def device_status(self) -> tuple[int, int]:
        return dec.dec_get_device_status(self.handle)

    def debug_dequant(self, layer: int, which: int, out: torch.Tensor) -> None:
        dec.dec_debug_dequant(self.handle, layer, which, _ptr(out), torch.cuda.current_stream().cuda_stream)

    def kernel_bytes(self, kernel_class: int, mean_cached_len: float) -> float:
        return dec.dec_kernel_bytes(self.handle, kernel_class, mean_cached_len)

    @property
    def launches_per_step(self) -> int:
        return dec.dec_launches_per_step(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            dec.dec_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

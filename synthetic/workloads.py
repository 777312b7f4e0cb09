"""Seeded synthetic inputs for the one-token decode step.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests.  It holds NO decoder arithmetic: it only draws random tensors with the
shapes and value distributions of the five workloads below (and of any custom
shape a test asks for), in a fixed, documented order, from a seeded
``torch.Generator``.

Workloads (shapes follow the Qwen3 family; values are random-init, there are
no trained weights):

* ``tiny``         2 layers, hidden 256, 4 q / 2 kv heads, head_dim 64,
                   intermediate 768, vocab 4096, bf16, batch 1, 128 cached
                   positions, 16 greedy steps, seed 0.
* ``qwen3-0.6b``   28 layers, hidden 1024, 16 q / 8 kv heads, head_dim 128,
                   intermediate 3072, vocab 151936, bf16, batch 1, 1024 cached
                   positions, 128 steps, seed 1.
* ``qwen3-4b-q4``  36 layers, hidden 2560, 32 q / 8 kv heads, head_dim 128,
                   intermediate 9728, vocab 151936, every linear (lm_head
                   included) affine 4-bit with groups of 64, batch 1, 4096
                   cached positions, 64 steps, seed 2.
* ``qwen3-8b-b8``  36 layers, hidden 4096, 32 q / 8 kv heads, head_dim 128,
                   intermediate 12288, vocab 151936, bf16, batch 8, 2048
                   cached positions each, 32 steps, seed 3.
* ``qwen3-8b-b1``  the same model at batch 1 (the single-stream case), seed 3.
* ``qwen3-8b-q4-b32`` the 8B shapes in the affine 4-bit format, batch 32,
                   cached lengths uniform in [512, 8192] per sequence, 32
                   steps, seed 4.
* ``*-kv8``        the same workload (same seed and draws up to the cache) with
                   the KV cache in the affine 8-bit format (``tiny-kv8``,
                   ``qwen3-8b-b1-kv8``, ``qwen3-8b-q4-b32-kv8``).

Value distributions: linear and embedding weights N(0, 0.02); norm weights
1 + N(0, 0.1); cached K/V N(0, 1); for 4-bit linears, uniform random 32-bit
words (so every nibble is uniform in 0..15), scales U(0.001, 0.01) and biases
N(0, 0.02).  Every floating value is drawn in fp32 and rounded to bf16 with
round-to-nearest-even (torch's conversion).  An affine 8-bit cache is drawn in
its stored form: codes uniform in 0..255, per group of 64 a scale U(0.015,
0.023) and a bias -scale * U(110, 145), both rounded to bf16 (values spread over
about [-2.8, 2.8] like a quantized N(0, 1) row).

Draw order: embed; per layer in_norm, q, k, v, o, q_norm, k_norm, post_norm,
gate, up, down; final_norm; lm_head; KV (layer by layer, K plane then V plane);
prompt tokens; cached lengths.  A 4-bit linear draws words, scales, biases; an
affine 8-bit cache draws, per layer and plane, codes, scales, bias factors.

Layouts (all row-major, linears are [out][in]):
  bf16 linear      int16/bfloat16 tensor [out, in]
  affine4 linear   dict(w=int32 [out, in/8] (nibble k of word j is input
                   element 8j+k, bits 4k..4k+3), scales=bf16 [out, in/64],
                   biases=bf16 [out, in/64])
  KV cache         bf16 [L][2][B][n_kv][max_ctx][head_dim]  (plane 0 = K,
                   plane 1 = V); affine 8-bit: dict(codes=uint8
                   [L][2][B][n_kv][max_ctx][head_dim], params=bf16
                   [L][2][B][n_kv][max_ctx][head_dim/64][2] (scale, bias))
"""

from __future__ import annotations

import dataclasses
from typing import Any

import torch

BF16 = "bf16"
AFFINE4_G64 = "affine4_g64"
AFFINE8_G64 = "affine8_g64"  # KV cache format
GROUP = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    weight_format: str
    batch: int
    prefill: int | tuple[int, int]  # fixed cached length, or inclusive uniform range
    steps: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    weight_std: float = 0.02
    norm_std: float = 0.1
    kv_format: str = BF16

    @property
    def max_prefill(self) -> int:
        return self.prefill[1] if isinstance(self.prefill, tuple) else self.prefill

    @property
    def max_ctx(self) -> int:
        """Cache slots per sequence: every cached position plus one per step (rounded up to
        a multiple of 16 for the affine 8-bit cache, which needs that)."""
        n = self.max_prefill + self.steps
        return (n + 15) // 16 * 16 if self.kv_format == AFFINE8_G64 else n

    def shapes(self) -> dict[str, tuple[int, int]]:
        H, d = self.hidden, self.head_dim
        return {
            "q": (self.n_q_heads * d, H),
            "k": (self.n_kv_heads * d, H),
            "v": (self.n_kv_heads * d, H),
            "o": (H, self.n_q_heads * d),
            "gate": (self.intermediate, H),
            "up": (self.intermediate, H),
            "down": (H, self.intermediate),
            "lm_head": (self.vocab, H),
        }

    def kv_shape(self) -> tuple[int, ...]:
        return (self.n_layers, 2, self.batch, self.n_kv_heads, self.max_ctx, self.head_dim)

    def replace(self, **kw: Any) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", 0, 2, 256, 4, 2, 64, 768, 4096, BF16, 1, 128, 16),
    "qwen3-0.6b": Workload("qwen3-0.6b", 1, 28, 1024, 16, 8, 128, 3072, 151936, BF16, 1, 1024, 128),
    "qwen3-4b-q4": Workload("qwen3-4b-q4", 2, 36, 2560, 32, 8, 128, 9728, 151936, AFFINE4_G64, 1, 4096, 64),
    "qwen3-8b-b8": Workload("qwen3-8b-b8", 3, 36, 4096, 32, 8, 128, 12288, 151936, BF16, 8, 2048, 32),
    "qwen3-8b-b1": Workload("qwen3-8b-b1", 3, 36, 4096, 32, 8, 128, 12288, 151936, BF16, 1, 2048, 32),
    "qwen3-8b-q4-b32": Workload("qwen3-8b-q4-b32", 4, 36, 4096, 32, 8, 128, 12288, 151936, AFFINE4_G64, 32,
                                (512, 8192), 32),
}
for _name in ("tiny", "qwen3-8b-b1", "qwen3-8b-q4-b32"):
    WORKLOADS[_name + "-kv8"] = WORKLOADS[_name].replace(name=_name + "-kv8", kv_format=AFFINE8_G64)


def _normal_bf16(g: torch.Generator, shape, std: float, mean: float, device) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


def _uniform_bf16(g: torch.Generator, shape, lo: float, hi: float, device) -> torch.Tensor:
    x = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return (x * (hi - lo) + lo).to(torch.bfloat16)


def _linear(g: torch.Generator, wl: Workload, out: int, inp: int, fmt: str, device):
    if fmt == BF16:
        return _normal_bf16(g, (out, inp), wl.weight_std, 0.0, device)
    assert inp % GROUP == 0, "affine 4-bit linears need in % 64 == 0"
    words = torch.randint(-(2 ** 31), 2 ** 31, (out, inp // 8), generator=g, device=device, dtype=torch.int64)
    words = words.to(torch.int32)
    scales = _uniform_bf16(g, (out, inp // GROUP), 0.001, 0.01, device)
    biases = _normal_bf16(g, (out, inp // GROUP), wl.weight_std, 0.0, device)
    return {"w": words, "scales": scales, "biases": biases}


def _kv_affine8(g: torch.Generator, wl: Workload, device) -> dict:
    shape = wl.kv_shape()
    codes = torch.empty(shape, dtype=torch.uint8, device=device)
    params = torch.empty(shape[:5] + (wl.head_dim // GROUP, 2), dtype=torch.bfloat16, device=device)
    for l in range(wl.n_layers):
        for p in range(2):
            codes[l, p].copy_(torch.randint(0, 256, shape[2:], generator=g, device=device, dtype=torch.int32))
            sc = torch.rand(params.shape[2:6], generator=g, device=device, dtype=torch.float32) * 0.008 + 0.015
            off = torch.rand(params.shape[2:6], generator=g, device=device, dtype=torch.float32) * 35.0 + 110.0
            sc16 = sc.to(torch.bfloat16)
            params[l, p, ..., 0].copy_(sc16)
            params[l, p, ..., 1].copy_((-sc16.float() * off).to(torch.bfloat16))
    return {"codes": codes, "params": params}


def kv_buffer(kv) -> torch.Tensor:
    """The cache as the one flat buffer the library reads: a bf16 cache as it is; an
    affine 8-bit cache as its codes, zero padding to a multiple of 256 bytes, then its
    (scale, bias) pairs."""
    if isinstance(kv, torch.Tensor):
        return kv
    codes = kv["codes"].reshape(-1)
    params = kv["params"].contiguous().view(torch.uint8).reshape(-1)
    pad = (-codes.numel()) % 256
    return torch.cat([codes, torch.zeros(pad, dtype=torch.uint8, device=codes.device), params])


def generate(wl: Workload, device: str | torch.device = "cpu", with_kv: bool = True) -> dict:
    """Draw the model, the prefilled KV cache and the first-step inputs of ``wl``.

    Returns a dict with ``embed``, ``final_norm``, ``lm_head``, ``layers`` (list
    of dicts), ``kv`` (or None), ``tokens`` int32 [B] and ``positions`` int32 [B]
    (the number of cached positions per sequence = the slot the next step writes).
    """
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed)
    sh = wl.shapes()
    fmt = wl.weight_format
    H, d = wl.hidden, wl.head_dim
    model: dict[str, Any] = {}
    model["embed"] = _normal_bf16(g, (wl.vocab, H), wl.weight_std, 0.0, device)
    layers = []
    for _ in range(wl.n_layers):
        lay: dict[str, Any] = {}
        lay["in_norm"] = _normal_bf16(g, (H,), wl.norm_std, 1.0, device)
        for name in ("q", "k", "v", "o"):
            lay[name] = _linear(g, wl, *sh[name], fmt, device)
        lay["q_norm"] = _normal_bf16(g, (d,), wl.norm_std, 1.0, device)
        lay["k_norm"] = _normal_bf16(g, (d,), wl.norm_std, 1.0, device)
        lay["post_norm"] = _normal_bf16(g, (H,), wl.norm_std, 1.0, device)
        for name in ("gate", "up", "down"):
            lay[name] = _linear(g, wl, *sh[name], fmt, device)
        layers.append(lay)
    model["layers"] = layers
    model["final_norm"] = _normal_bf16(g, (H,), wl.norm_std, 1.0, device)
    model["lm_head"] = _linear(g, wl, *sh["lm_head"], fmt, device)

    if with_kv and wl.kv_format == AFFINE8_G64:
        model["kv"] = _kv_affine8(g, wl, device)
    elif with_kv:
        kv = torch.empty(wl.kv_shape(), dtype=torch.bfloat16, device=device)
        for l in range(wl.n_layers):
            for p in range(2):
                kv[l, p].copy_(_normal_bf16(g, kv.shape[2:], 1.0, 0.0, device))
        model["kv"] = kv
    else:
        model["kv"] = None

    model["tokens"] = torch.randint(0, wl.vocab, (wl.batch,), generator=g, device=device,
                                    dtype=torch.int64).to(torch.int32)
    if isinstance(wl.prefill, tuple):
        lo, hi = wl.prefill
        pos = torch.randint(lo, hi + 1, (wl.batch,), generator=g, device=device, dtype=torch.int64)
    else:
        pos = torch.full((wl.batch,), wl.prefill, device=device, dtype=torch.int64)
    model["positions"] = pos.to(torch.int32)
    return model


def custom(name: str = "custom", **kw: Any) -> Workload:
    """A small workload with explicit shapes, for edge-case tests."""
    base = dict(seed=123, n_layers=1, hidden=128, n_q_heads=2, n_kv_heads=1, head_dim=64,
                intermediate=256, vocab=512, weight_format=BF16, batch=1, prefill=16, steps=2)
    base.update(kw)
    return Workload(name=name, **base)


def to_host(model: dict) -> dict:
    """Copy every tensor of a generated model to host memory (same dtypes)."""
    def mv(x):
        if isinstance(x, torch.Tensor):
            return x.cpu()
        if isinstance(x, dict):
            return {k: mv(v) for k, v in x.items()}
        if isinstance(x, list):
            return [mv(v) for v in x]
        return x
    return mv(model)

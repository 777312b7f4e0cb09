"""CPU oracle for the one-token decode step of a Qwen3-style dense decoder.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, float64 numpy
statement of what one decode step computes.  It shares no code, header, table
or constant generator with the CUDA library under ``token_decode_step_gb300``
and never imports it.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it;
the product path never does.

Sources (page title and section):
  * ANEForge, "LLMs on the ANE": section "What's inside" (pre-norm block order
    RMSNorm -> QKV -> RoPE -> GQA causal attention -> SwiGLU MLP with
    residuals; RoPE as x*cos + rotate_half(x)*sin; KV heads shared by groups of
    query heads) and section "Correctness" (Qwen3: separate head_dim, per-head
    RMSNorm on Q and K before RoPE); section "lm_head on the ANE" (tiling the
    vocab; the top-2 tie margin).
  * Butter architecture ("architecture.md", FFAI planning): figure
    "SINGLE-TOKEN DECODE" (gather, rms_norm, q/k/v gemv, rope at offset =
    cache length, cache append into a preallocated buffer, sdpa_decode, o
    gemv + add, rms_norm, gate/up gemv, silu_mul, down gemv + add, final
    rms_norm, lm_head gemv) and section on GPU sampling (greedy = argmax over
    the vocab axis).
  * The same Butter section on GPU sampling for oracle/sampling.py: temperature,
    top-k, top-p, then an inverse-CDF draw from a counter-based generator
    (Philox4x32-10 from its publication; its known-answer vectors pin it).
  * oxinfer (docs.rs crate page), section "MLX checkpoints": packed 4-bit
    weights, eight per uint32, bf16 scale and bias per group of 64,
    w = scale * q + bias.
  * Butter architecture.md, model-layer section (per-layer cache types include an
    AffineQuantizedKVCache) for oracle/kvcache.py: the cache may hold affine 8-bit
    codes with a bf16 scale and bias per group of 64 instead of bf16 rows.

Readings where the pages are silent:
  * RoPE pairs element i with element i + d/2 (rotate-half), angle
    pos * theta^(-2i/d), theta = 1e6.
  * RMSNorm multiplies by the stored weight w (not 1 + w), eps = 1e-6; the q/k
    norm weight has shape [head_dim] and is shared by all heads of a layer.
  * Nibble k of packed word j is input element 8j + k, bits 4k..4k+3.
  * The new token attends to cached slots 0..P inclusive (P = cached length),
    after its own K/V were written at slot P; scale 1/sqrt(head_dim).
  * The cache stores bf16: the appended K and V are rounded to bf16
    (round-to-nearest-even) before they are used; or, in the affine 8-bit format,
    they are quantized (min-max per group of 64, decisions in float32, see
    oracle/kvcache.py) and read back as scale * code + bias.
  * argmax ties go to the lowest index.

Parity-unpinned pieces: none of the functions below lacks a pin (see
tests/test_oracle_pins.py); the end-to-end step values themselves have no
worked example on the pages and are pinned by composition of the pinned parts
plus an independent scalar-loop restatement on a tiny shape.
"""

from .numerics import bf16_bits_to_f64, f64_to_bf16_bits, round_to_bf16  # noqa: F401
from .affine4 import dequant_affine4_g64, dequant_affine4_g64_f32  # noqa: F401
from . import sampling  # noqa: F401
from .kvcache import Affine8Cache, quantize_affine8_g64, dequant_affine8_g64  # noqa: F401
from .decoder import (  # noqa: F401
    OracleModel, rmsnorm, rope_rotate_half, softmax, gqa_attention, lse_merge, silu,
    argmax_lowest, decode_step, tie_exempt, verify_step,
)

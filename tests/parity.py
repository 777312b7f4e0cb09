"""Helpers for the GPU parity tests: run the CUDA step through the C ABI, replay
the oracle on the same seeded inputs, compare with the stated tolerances.

Tolerances (per step, per sequence, over the vocab): max |logit diff| <= 5e-2 and
||diff||_2 / ||ref||_2 <= 1e-2; the argmax must be equal unless the oracle's top-2
gap is below 1e-2 * max|logit| (near tie).
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import synthetic
from oracle import numerics

MAX_ABS = 5e-2
REL_L2 = 1e-2
TIE_REL = 1e-2

# attention-kernel output tolerance: max |out - ref| <= ATTN_ATOL + ATTN_RTOL * |ref|.
# The kernel keeps ~16 significant bits of q and of the probabilities (bf16 hi + lo)
# with fp32 accumulation, so its error is ~1e-6 of the value scale.
ATTN_ATOL, ATTN_RTOL = 1e-4, 1e-4


def np_model(model: dict) -> dict:
    def conv(x):
        if isinstance(x, dict):
            return {k: conv(v) for k, v in x.items()}
        if isinstance(x, list):
            return [conv(v) for v in x]
        if x is None:
            return None
        return oracle.decoder._to_numpy(x)
    return {k: conv(v) for k, v in model.items()}


def check_logits(gpu: np.ndarray, ref: np.ndarray, gpu_argmax, ref_argmax, where: str = "") -> dict:
    """Assert the tolerance rule for every sequence; returns the worst errors seen."""
    worst = {"max_abs": 0.0, "rel_l2": 0.0, "exempt": 0}
    for b in range(ref.shape[0]):
        d = gpu[b].astype(np.float64) - ref[b]
        ma = float(np.max(np.abs(d)))
        rl = float(np.linalg.norm(d) / np.linalg.norm(ref[b]))
        worst["max_abs"] = max(worst["max_abs"], ma)
        worst["rel_l2"] = max(worst["rel_l2"], rl)
        assert ma <= MAX_ABS, f"{where} seq {b}: max|dlogit| {ma:.3e} > {MAX_ABS}"
        assert rl <= REL_L2, f"{where} seq {b}: rel L2 {rl:.3e} > {REL_L2}"
        if int(gpu_argmax[b]) != int(ref_argmax[b]):
            assert oracle.tie_exempt(ref[b], TIE_REL), (
                f"{where} seq {b}: argmax {int(gpu_argmax[b])} != oracle {int(ref_argmax[b])} outside the tie margin")
            worst["exempt"] += 1
    return worst


def gpu_greedy(dec_obj, model_dev: dict, steps: int, want_logits: bool = True):
    """Greedy loop on the device: tokens <- argmax, positions += 1 after every step.
    Returns per-step (input tokens, input positions, logits, argmax) on the host and
    the final KV cache (device tensor)."""
    B = dec_obj.cfg.batch
    V = dec_obj.cfg.vocab
    tokens = model_dev["tokens"].clone()
    positions = model_dev["positions"].clone()
    kv = model_dev["kv"]
    logits = torch.empty((B, V), dtype=torch.float32, device="cuda") if want_logits else None
    argmax = torch.empty((B,), dtype=torch.int32, device="cuda")
    out = []
    for _ in range(steps):
        tin, pin = tokens.cpu().numpy().copy(), positions.cpu().numpy().copy()
        dec_obj.step(tokens, positions, kv, logits, argmax)
        torch.cuda.synchronize()
        out.append((tin, pin, logits.cpu().numpy().copy() if want_logits else None, argmax.cpu().numpy().copy()))
        dec_obj.advance(argmax, tokens, positions)
    torch.cuda.synchronize()
    return out, kv


def select_seqs(kv, seqs):
    """The oracle-side cache of the sequences `seqs` (a copy): bf16 bit patterns
    [L][2][B][...] or an affine 8-bit cache, sliced along the batch axis."""
    if seqs is None:
        return kv.copy()
    idx = np.asarray(seqs)
    if isinstance(kv, np.ndarray):
        return kv[:, :, idx].copy()
    return oracle.Affine8Cache(kv.codes[:, :, idx].copy(), kv.params[:, :, idx].copy())


def oracle_replay(wl, model_host: dict, kv_init, gpu_steps, check_steps=None, cache_weights: bool = True,
                  seqs=None, model=None):
    """Replay the oracle on the GPU's token sequence (each side keeps its own KV).

    seqs: the sequences to replay (None: the whole batch).  The sequences of a batch are
    independent (own token, cache and position), so a subset replays exactly what the
    batched step computed for them.  Returns ([(step, oracle logits [len(seqs)][V],
    oracle argmax)] for the checked steps, final oracle KV of those sequences); every
    step up to the last checked one is computed, since the KV state depends on all of
    them.  `model`: an OracleModel to reuse (its float64 weights already converted)."""
    m = model if model is not None else oracle.OracleModel.from_synthetic(wl, model_host,
                                                                          cache_weights=cache_weights)
    kv = select_seqs(kv_init, seqs)
    sel = slice(None) if seqs is None else np.asarray(seqs)
    last = max(check_steps) if check_steps else len(gpu_steps) - 1
    res = []
    for s, (tin, pin, _, _) in enumerate(gpu_steps[: last + 1]):
        logits, am = oracle.decode_step(m, kv, tin[sel], pin[sel])
        if check_steps is None or s in check_steps:
            res.append((s, logits, am))
    return res, kv


def replay_plan(wl):
    """Which (sequences, steps) the full-size step tests replay in the oracle.

    Every config is replayed over ALL of its greedy steps.  Batches above 4 sequences are
    replayed over all steps for 3 fixed sequences (the first, the middle one and the last)
    and, for every sequence, over the first 2 steps.  Returns a list of (seqs or None, steps)."""
    if wl.batch <= 4:
        return [(None, wl.steps)]
    fixed = sorted({0, wl.batch // 2, wl.batch - 1})
    return [(fixed, wl.steps), (None, 2)]


def kv_appended_close(gpu_kv: np.ndarray, ref_kv: np.ndarray, kv_init: np.ndarray) -> None:
    """Untouched cache slots must be bit-identical.  Every appended K or V vector
    (one head, one position) must match the oracle's to within two bf16 steps at
    the vector's own scale: max |gpu - ref| <= 2 * 2^-8 * max |ref|.  (fp32 versus
    float64 accumulation over many layers moves near-zero elements by more than
    their own ulp, but stays far below the quantisation step of the vector.)"""
    L, _, B, nkv, T, d = gpu_kv.shape
    changed = np.any((gpu_kv != kv_init) | (ref_kv != kv_init), axis=-1)  # [L,2,B,nkv,T]
    assert np.array_equal(gpu_kv[~changed], kv_init[~changed])
    idx = np.argwhere(changed)
    g = numerics.bf16_bits_to_f64(gpu_kv[changed])   # [n, d]
    r = numerics.bf16_bits_to_f64(ref_kv[changed])
    scale = np.max(np.abs(r), axis=-1)
    err = np.max(np.abs(g - r), axis=-1)
    bad = err > 2 * 2.0 ** -8 * scale
    if np.any(bad):
        worst = np.argsort(-(err / np.maximum(scale, 1e-30)))[:5]
        rows = [f"{tuple(int(v) for v in idx[i])}: max err {err[i]:.3g} scale {scale[i]:.3g}" for i in worst]
        raise AssertionError(f"{int(bad.sum())} of {len(err)} appended K/V vectors differ by more than 2 bf16 "
                             f"steps: " + "; ".join(rows))


def make_attention_case(seed, B, nq, nkv, d, positions, max_ctx, n_layers=2):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    qkv = torch.randn((B, (nq + 2 * nkv) * d), generator=g) * 0.7
    q_norm = (1 + 0.1 * torch.randn((d,), generator=g)).to(torch.bfloat16)
    k_norm = (1 + 0.1 * torch.randn((d,), generator=g)).to(torch.bfloat16)
    kv = torch.randn((n_layers, 2, B, nkv, max_ctx, d), generator=g).to(torch.bfloat16)
    pos = torch.tensor(positions, dtype=torch.int32)
    return qkv, q_norm, k_norm, kv, pos


def attention_cfg(dec, B, nq, nkv, d, max_ctx, n_layers=2):
    return dec.DecConfig(n_layers=n_layers, hidden=64, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, intermediate=64,
                         vocab=1, rms_eps=1e-6, rope_theta=1e6, linear_fmt=0, batch=B, max_ctx=max_ctx)

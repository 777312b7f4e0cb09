"""One decode step of a Qwen3-style dense decoder, in float64 (test infrastructure only).

Every function states the computation plainly; nothing is fused, tiled or
reordered.  Page citations are by page title and section:

  [ANE-inside]   ANEForge "LLMs on the ANE", section "What's inside"
  [ANE-correct]  ANEForge "LLMs on the ANE", section "Correctness"
  [ANE-head]     ANEForge "LLMs on the ANE", section "lm_head on the ANE"
  [Butter-decode] Butter architecture.md, figure "SINGLE-TOKEN DECODE"
  [Butter-sample] Butter architecture.md, GPU sampling figure (greedy argmax)
  [oxi-mlx]      oxinfer crate page, section "MLX checkpoints"
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .affine4 import dequant_affine4_g64
from .kvcache import Affine8Cache, kv_read, kv_store
from .numerics import bf16_bits_to_f64


# --------------------------------------------------------------------------- ops

def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w over the last axis [Butter-decode rms_norm;
    Qwen uses the plain weight w]."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_rotate_half(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotary embedding at position ``pos`` [ANE-inside: x*cos + rotate_half(x)*sin].

    x has head_dim d on its last axis.  For i < d/2 the angle is
    pos * theta**(-2i/d); rotate_half(x) = concat(-x[d/2:], x[:d/2]); the
    cos/sin vectors repeat the d/2 angles twice.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    ang = pos * theta ** (-2.0 * i / d)
    cos = np.concatenate([np.cos(ang), np.cos(ang)])
    sin = np.concatenate([np.sin(ang), np.sin(ang)])
    rot = np.concatenate([-x[..., half:], x[..., :half]], axis=-1)
    return x * cos + rot * sin


def softmax(s: np.ndarray) -> np.ndarray:
    """exp(s - max) / sum(exp(s - max)) over the last axis."""
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    return e / np.sum(e, axis=-1, keepdims=True)


def gqa_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Decode attention for one sequence [Butter-decode sdpa_decode; ANE-inside GQA].

    q [n_q, d]; K, V [n_kv, T, d] hold every position the new token may see
    (its own included).  Query head j reads KV head j // (n_q / n_kv); the
    scores q.K^T are scaled by 1/sqrt(d) and soft-maxed over the T positions.
    """
    n_q, d = q.shape
    n_kv = K.shape[0]
    assert n_q % n_kv == 0
    group = n_q // n_kv
    out = np.empty((n_q, d), dtype=np.float64)
    for j in range(n_q):
        h = j // group
        s = (K[h] @ q[j]) / np.sqrt(d)
        p = softmax(s)
        out[j] = p @ V[h]
    return out


def attention_partial(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> tuple[float, float, np.ndarray]:
    """Un-normalised softmax statistics of one head over a subset of positions:
    (m, l, acc) with m = max score, l = sum exp(s - m), acc = sum exp(s - m) v."""
    d = q.shape[-1]
    s = (K @ q) / np.sqrt(d)
    m = float(np.max(s))
    e = np.exp(s - m)
    return m, float(np.sum(e)), e @ V


def lse_merge(parts: list[tuple[float, float, np.ndarray]]) -> np.ndarray:
    """Combine partial softmax statistics of disjoint position subsets:
    o = sum_i e^(m_i - M) acc_i / sum_i e^(m_i - M) l_i with M = max_i m_i.
    (The merge identity used by split-KV decoding; pinned against one-pass
    softmax in the oracle tests.)"""
    M = max(p[0] for p in parts)
    num = sum(np.exp(p[0] - M) * p[2] for p in parts)
    den = sum(np.exp(p[0] - M) * p[1] for p in parts)
    return num / den


def silu(x: np.ndarray) -> np.ndarray:
    """x / (1 + e^-x) [Butter-decode silu_mul]."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def argmax_lowest(x: np.ndarray) -> int:
    """Index of the maximum, the lowest one among equal maxima [Butter-sample]."""
    x = np.asarray(x)
    m = np.max(x)
    return int(np.flatnonzero(x == m)[0])


def tie_exempt(logits: np.ndarray, rel: float = 1e-2) -> bool:
    """True when the top-2 gap is below rel * max|logit|: a near tie whose argmax
    may legitimately differ between two correct implementations (the tie-margin
    notion of [ANE-head], with the tolerance of this project)."""
    top2 = np.sort(np.asarray(logits, dtype=np.float64))[-2:]
    return bool(top2[1] - top2[0] < rel * np.max(np.abs(logits)))


# ------------------------------------------------------------------------- model

def _to_numpy(t):
    """torch tensor / numpy array -> numpy (bf16 tensors become uint16 bit patterns)."""
    if isinstance(t, np.ndarray):
        return t
    import torch  # only for unpacking the synthetic inputs
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.int32:
        return t.cpu().numpy()
    return t.cpu().numpy()


@dataclass
class OracleModel:
    """Host copy of a synthetic model with lazily converted float64 weights."""
    cfg: object  # synthetic.Workload-like: shapes, eps, theta
    raw: dict
    cache_weights: bool = True
    _cache: dict = field(default_factory=dict)

    @classmethod
    def from_synthetic(cls, cfg, model: dict, cache_weights: bool = True) -> "OracleModel":
        def conv(x):
            if isinstance(x, dict):
                return {k: conv(v) for k, v in x.items()}
            if isinstance(x, list):
                return [conv(v) for v in x]
            if x is None:
                return None
            return _to_numpy(x)
        raw = {k: conv(v) for k, v in model.items() if k not in ("kv", "tokens", "positions")}
        return cls(cfg, raw, cache_weights)

    def vec(self, *path) -> np.ndarray:
        key = ("vec",) + path
        if key not in self._cache:
            node = self.raw
            for p in path:
                node = node[p]
            self._cache[key] = bf16_bits_to_f64(node)
        return self._cache[key]

    def matrix(self, *path) -> np.ndarray:
        """float64 weight matrix [out, in] of a linear (bf16 or affine 4-bit)."""
        key = ("mat",) + path
        if key in self._cache:
            return self._cache[key]
        node = self.raw
        for p in path:
            node = node[p]
        if isinstance(node, dict):
            w = dequant_affine4_g64(node["w"].view(np.uint32), node["scales"], node["biases"])
        else:
            w = bf16_bits_to_f64(node)
        if self.cache_weights:
            self._cache[key] = w
        return w

    def linear(self, x: np.ndarray, *path) -> np.ndarray:
        """y = W x for x [..., in] (rows of x are independent sequences)."""
        return x @ self.matrix(*path).T

    def embed_row(self, tok: int) -> np.ndarray:
        return bf16_bits_to_f64(self.raw["embed"][tok])


def decode_step(m: OracleModel, kv: np.ndarray, tokens, positions):
    """One greedy decode step for B independent sequences.

    kv: uint16 bf16 bit patterns [L][2][B][n_kv][max_ctx][d], or an Affine8Cache;
    slot P_b of every layer is overwritten with the new token's K and V in the
    cache's format (rounded to bf16, or quantized to affine 8-bit codes).
    tokens[b]: input token id; positions[b] = P_b = number of cached positions.
    Returns (logits float64 [B, V], argmax int64 [B]).

    Block order [ANE-inside; Butter-decode]:
      h = embed[token]
      per layer: xn = rms(h, in_norm); q,k,v = Wq xn, Wk xn, Wv xn;
                 per-head rms on q (q_norm) and k (k_norm) before RoPE [ANE-correct];
                 RoPE at position P; append k,v at slot P; attend over 0..P;
                 h += Wo o; xn = rms(h, post_norm); h += Wdown(silu(Wgate xn) * Wup xn)
      logits = Wlm rms(h, final_norm); argmax over the vocab (lowest index on ties).
    """
    cfg = m.cfg
    L, nq, nkv, d = cfg.n_layers, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    eps, theta = cfg.rms_eps, cfg.rope_theta
    tokens = [int(t) for t in np.asarray(tokens).reshape(-1)]
    positions = [int(p) for p in np.asarray(positions).reshape(-1)]
    B = len(tokens)
    assert kv.shape[:3] == (L, 2, B)
    assert isinstance(kv, Affine8Cache) or kv.dtype == np.uint16
    for P in positions:
        assert 0 <= P < kv.shape[4], "position outside the cache"

    h = np.stack([m.embed_row(t) for t in tokens])  # [B, H]
    for l in range(L):
        xn = rmsnorm(h, m.vec("layers", l, "in_norm"), eps)
        q = m.linear(xn, "layers", l, "q").reshape(B, nq, d)
        k = m.linear(xn, "layers", l, "k").reshape(B, nkv, d)
        v = m.linear(xn, "layers", l, "v").reshape(B, nkv, d)
        q = rmsnorm(q, m.vec("layers", l, "q_norm"), eps)
        k = rmsnorm(k, m.vec("layers", l, "k_norm"), eps)
        o = np.empty((B, nq * d), dtype=np.float64)
        for b in range(B):
            P = positions[b]
            qb = rope_rotate_half(q[b], P, theta)
            kb = rope_rotate_half(k[b], P, theta)
            kv_store(kv, l, 0, b, P, kb)
            kv_store(kv, l, 1, b, P, v[b])
            Kc = kv_read(kv, l, 0, b, P + 1)
            Vc = kv_read(kv, l, 1, b, P + 1)
            o[b] = gqa_attention(qb, Kc, Vc).reshape(-1)
        h = h + m.linear(o, "layers", l, "o")
        xn = rmsnorm(h, m.vec("layers", l, "post_norm"), eps)
        g = silu(m.linear(xn, "layers", l, "gate")) * m.linear(xn, "layers", l, "up")
        h = h + m.linear(g, "layers", l, "down")
    logits = m.linear(rmsnorm(h, m.vec("final_norm"), eps), "lm_head")
    am = np.array([argmax_lowest(logits[b]) for b in range(B)], dtype=np.int64)
    return logits, am


def verify_step(m: OracleModel, kv: np.ndarray, tokens, positions):
    """Multi-token verify step (speculative decoding's check of drafted tokens): for
    each sequence b, tokens[b][0..T-1] at positions P_b .. P_b + T - 1.  Row (b, t) is,
    by definition, the one-token step of sequence b at position P_b + t after the rows
    (b, 0..t-1) were appended: T decode steps with the given tokens fed in (teacher
    forcing), each appending its K/V.  Returns (logits float64 [B, T, V], argmax int64
    [B, T]).  Sources: ANEForge "LLMs on the ANE", section "Speculative decoding" (a
    draft proposes K tokens, the target verifies all K in one forward); Butter
    architecture.md, phase 8 speculative decoding (one verifier pass scores all K
    candidates, batched along the sequence)."""
    tokens = np.asarray(tokens)
    positions = np.asarray(positions)
    T = tokens.shape[1]
    logits, am = [], []
    for t in range(T):
        lg, a = decode_step(m, kv, tokens[:, t], positions + t)
        logits.append(lg)
        am.append(a)
    return np.stack(logits, axis=1), np.stack(am, axis=1)

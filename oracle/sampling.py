"""On-device sampling, stated plainly (TEST INFRASTRUCTURE ONLY, see the package header).

Source: Butter architecture ("architecture.md", FFAI planning), section on GPU
sampling: after the lm_head the sampling kernel reads the logits on the device and
applies, in order, temperature (logits times 1/temp), top-k (sort, keep the k
largest, mask the rest), top-p (cumulative softmax, threshold mask) and an
inverse-CDF draw with an RNG state; greedy (temperature 0) is the argmax.  oxinfer's
crate page lists the same knobs (--temp, --top-k, --top-p, --seed).

Readings where the page is silent:
  * Candidates: the k largest logits under the total order (logit descending, index
    ascending), k = top_k for 1 <= top_k <= 1024, else 1024 (the page sorts "top k";
    a sort of the whole vocabulary has no counterpart).  k is at most the vocabulary.
  * The candidates stay in that order; p_j = exp((l_j - l_0) / temperature).
  * top-p keeps the shortest prefix whose cumulative mass reaches top_p of the
    candidates' mass (top_p >= 1 keeps all k).
  * The draw: u in [0, 1) from Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
    "Parallel random numbers: as easy as 1, 2, 3", SC'11) with key (seed low 32 bits,
    seed high 32 bits) and counter (offset low, offset high, row, 0); u = (x0 >> 8)
    * 2^-24 from the first output word.  The token is the first candidate of the
    kept prefix whose cumulative mass exceeds u times the prefix's mass.
  * Temperature 0 (or below): the argmax, lowest index on ties.

The arithmetic here is float64 on the float32 logits; the candidate set depends only
on comparisons of the float32 inputs and is therefore exact.
"""

from __future__ import annotations

import math

import numpy as np

K_MAX = 1024
_M0, _M1 = 0xD2511F53, 0xCD9E8D57
_W0, _W1 = 0x9E3779B9, 0xBB67AE85
_MASK = 0xFFFFFFFF


def philox4x32_10(counter: tuple[int, int, int, int], key: tuple[int, int]) -> tuple[int, int, int, int]:
    """Ten rounds of Philox-4x32: each round multiplies words 0 and 2 by the two
    round multipliers (64-bit products split into high and low halves), mixes the
    high halves with words 1 and 3 and the round key, and permutes; the key is
    advanced by the two Weyl constants after every round."""
    c0, c1, c2, c3 = (int(x) & _MASK for x in counter)
    k0, k1 = (int(x) & _MASK for x in key)
    for _ in range(10):
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> 32, p0 & _MASK
        hi1, lo1 = p1 >> 32, p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & _MASK, lo1, (hi0 ^ c3 ^ k1) & _MASK, lo0
        k0 = (k0 + _W0) & _MASK
        k1 = (k1 + _W1) & _MASK
    return c0, c1, c2, c3


def uniform24(seed: int, offset: int, row: int) -> float:
    """u in [0, 1) with 24 random bits: exactly representable in float32 too."""
    x0 = philox4x32_10((offset & _MASK, (offset >> 32) & _MASK, row & _MASK, 0), (seed & _MASK, (seed >> 32) & _MASK))[0]
    return (x0 >> 8) * 2.0 ** -24


def candidates(logits_f32: np.ndarray, top_k: int) -> np.ndarray:
    """Indices of the k largest logits, ordered by (logit descending, index ascending)."""
    v = np.asarray(logits_f32, dtype=np.float32)
    k = top_k if 1 <= top_k <= K_MAX else K_MAX
    k = min(k, v.shape[0])
    # stable sort on the negated value keeps ascending indices among equal logits
    order = np.argsort(-v.astype(np.float64), kind="stable")
    return order[:k]


def sample_row(logits_f32: np.ndarray, temperature: float, top_k: int, top_p: float, u: float) -> dict:
    """The sampled token of one row, with the margins of the two decisions that floating
    point takes (top-p cut and draw) relative to the kept mass, for tie exemptions."""
    v = np.asarray(logits_f32, dtype=np.float32)
    if not temperature > 0.0:
        best = int(np.argmax(v))  # first occurrence of the maximum
        return {"token": best, "cut": None, "draw": None, "kept": 1, "cut_margin": math.inf,
                "draw_margin": math.inf}
    cand = candidates(v, top_k)
    lv = v[cand].astype(np.float64)
    t = float(np.float32(temperature))
    p = np.exp((lv - lv[0]) / t)
    cum = np.cumsum(p)
    total = cum[-1]
    if top_p < 1.0:
        thr = float(np.float32(top_p)) * total
        m = int(np.argmax(cum >= thr)) + 1
        cut_margin = float(np.min(np.abs(cum - thr))) / total
    else:
        m = len(cand)
        cut_margin = math.inf
    target = u * cum[m - 1]
    j = int(np.argmax(cum[:m] > target))
    draw_margin = float(np.min(np.abs(cum[:m] - target))) / cum[m - 1]
    return {"token": int(cand[j]), "kept": m, "cut_margin": cut_margin, "draw_margin": draw_margin,
            "candidates": cand, "cum": cum}


def sample(logits_f32: np.ndarray, temperature: float, top_k: int, top_p: float, seed: int, offset: int) -> list:
    """sample_row for every row of a [B, V] float32 array, u from (seed, offset, row)."""
    rows = np.asarray(logits_f32, dtype=np.float32)
    return [sample_row(rows[b], temperature, top_k, top_p, uniform24(seed, offset, b)) for b in range(rows.shape[0])]

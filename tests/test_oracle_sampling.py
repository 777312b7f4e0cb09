"""Pins of the oracle's sampler (oracle/sampling.py) against what the algorithm and the
mathematics fix: the Philox known-answer vectors, brute-force top-k order, the minimal
top-p prefix, and the inverse CDF reproducing the kept distribution exactly on a grid
of u values."""

import pathlib

import numpy as np
import pytest

from oracle import sampling as S

GOLDEN = pathlib.Path(__file__).parent / "golden" / "philox4x32_10_kat.txt"


def test_philox_known_answer_vectors():
    rows = [ln.split() for ln in GOLDEN.read_text().splitlines() if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        vals = [int(x, 16) for x in r]
        assert S.philox4x32_10(tuple(vals[0:4]), tuple(vals[4:6])) == tuple(vals[6:10])


def test_uniform24_range_and_grid():
    us = [S.uniform24(7, o, b) for o in range(50) for b in range(4)]
    assert all(0.0 <= u < 1.0 for u in us)
    assert all(u * 2**24 == int(u * 2**24) for u in us)
    assert len(set(us)) == len(us)  # distinct draws for distinct counters
    # the seed and the offset high word enter the key and the counter
    assert S.uniform24(1, 0, 0) != S.uniform24(1 << 32, 0, 0)
    assert S.uniform24(1, 1 << 32, 0) != S.uniform24(1, 0, 0)


def _brute_candidates(v, k):
    order = sorted(range(len(v)), key=lambda i: (-float(v[i]), i))
    return order[: min(k if 1 <= k <= S.K_MAX else S.K_MAX, len(v))]


@pytest.mark.parametrize("k", [1, 5, 64, 0, 2000])
def test_candidates_match_brute_force_with_ties(k):
    rng = np.random.default_rng(k + 3)
    v = rng.integers(-20, 20, size=3000).astype(np.float32) / 4  # many exact ties
    assert list(S.candidates(v, k)) == _brute_candidates(v, k)


def test_greedy_special_cases():
    rng = np.random.default_rng(0)
    v = rng.standard_normal(5000).astype(np.float32)
    v[4321] = v.max() + 1.0
    for u in (0.0, 0.3, 0.999):
        assert S.sample_row(v, 0.0, 0, 1.0, u)["token"] == 4321          # temperature 0
        assert S.sample_row(v, 0.7, 1, 1.0, u)["token"] == 4321          # top-k 1
        assert S.sample_row(v, 0.7, 50, 1e-9, u)["token"] == 4321        # top-p ~ 0 keeps one
    assert S.sample_row(v, 0.7, 50, 1.0, 0.0)["token"] == 4321           # u = 0: the first candidate


def test_top_p_prefix_is_minimal():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(4000) * 2).astype(np.float32)
    for top_p in (0.1, 0.5, 0.9, 0.99):
        r = S.sample_row(v, 0.8, 300, top_p, 0.5)
        cum, m = r["cum"], r["kept"]
        total = cum[-1]
        assert cum[m - 1] >= np.float32(top_p) * total
        assert m == 1 or cum[m - 2] < np.float32(top_p) * total


@pytest.mark.parametrize("temperature,top_k,top_p", [(1.0, 8, 1.0), (0.5, 20, 0.9), (2.0, 1024, 1.0)])
def test_inverse_cdf_reproduces_the_kept_distribution(temperature, top_k, top_p):
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(3000) * 1.5).astype(np.float32)
    ref = S.sample_row(v, temperature, top_k, top_p, 0.0)
    cand, m = ref["candidates"], ref["kept"]
    lv = v[cand[:m]].astype(np.float64)
    p = np.exp((lv - lv[0]) / np.float32(temperature))
    p /= p.sum()
    n = 20000
    counts = {}
    for i in range(n):
        tok = S.sample_row(v, temperature, top_k, top_p, (i + 0.5) / n)["token"]
        counts[tok] = counts.get(tok, 0) + 1
    assert set(counts) <= set(int(c) for c in cand[:m])
    for j, c in enumerate(cand[:m]):
        assert abs(counts.get(int(c), 0) / n - p[j]) <= 1.0 / n + 1e-12


def test_temperature_scales_log_probabilities():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(500).astype(np.float32)
    a = S.sample_row(v, 0.5, 10, 1.0, 0.25)
    b = S.sample_row((v.astype(np.float64) / 0.5).astype(np.float32), 1.0, 10, 1.0, 0.25)
    assert list(a["candidates"]) == list(b["candidates"])
    np.testing.assert_allclose(a["cum"] / a["cum"][-1], b["cum"] / b["cum"][-1], rtol=1e-6)

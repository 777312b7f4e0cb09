"""Whole-step checks of the oracle: an independent scalar-loop restatement on
tiny shapes, plus cache, causality and batch-independence invariants."""

import math

import numpy as np
import pytest

import oracle
import synthetic
from oracle import numerics


def _bf(bits):
    return float(numerics.bf16_bits_to_f64(np.array([bits], dtype=np.uint16))[0])


def _scalar_step(wl, model, kv, tokens, positions, kv_out=None):
    """A second statement of the decode step with Python scalars and loops only
    (no numpy linear algebra, no shared helper besides bf16 bit reading).  With kv_out,
    the new token's bf16 K and V bits are also written at slot P of every layer there."""
    L, H, nq, nkv, d, I, V = (wl.n_layers, wl.hidden, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                              wl.intermediate, wl.vocab)
    eps, theta = wl.rms_eps, wl.rope_theta
    group = nq // nkv

    def weight(lin, r, c):
        if isinstance(lin, dict):
            word = int(lin["w"][r, c // 8]) & 0xFFFFFFFF
            q = (word >> (4 * (c % 8))) & 15
            return _bf(lin["scales"][r, c // 64]) * q + _bf(lin["biases"][r, c // 64])
        return _bf(lin[r, c])

    def matvec(lin, x, n_out):
        return [sum(weight(lin, r, c) * x[c] for c in range(len(x))) for r in range(n_out)]

    def norm(x, w):
        ms = sum(v * v for v in x) / len(x)
        inv = 1.0 / math.sqrt(ms + eps)
        return [x[i] * inv * _bf(w[i]) for i in range(len(x))]

    def rope(x, pos):
        half = d // 2
        y = [0.0] * d
        for i in range(half):
            a = pos * theta ** (-2.0 * i / d)
            y[i] = x[i] * math.cos(a) - x[i + half] * math.sin(a)
            y[i + half] = x[i + half] * math.cos(a) + x[i] * math.sin(a)
        return y

    out_logits = []
    for b in range(len(tokens)):
        P = int(positions[b])
        h = [_bf(v) for v in model["embed"][int(tokens[b])]]
        for l in range(L):
            lay = model["layers"][l]
            xn = norm(h, lay["in_norm"])
            q = matvec(lay["q"], xn, nq * d)
            k = matvec(lay["k"], xn, nkv * d)
            v = matvec(lay["v"], xn, nkv * d)
            qh = [rope(norm(q[j * d:(j + 1) * d], lay["q_norm"]), P) for j in range(nq)]
            kh = [rope(norm(k[j * d:(j + 1) * d], lay["k_norm"]), P) for j in range(nkv)]
            vh = [v[j * d:(j + 1) * d] for j in range(nkv)]
            # keys/values the new token sees: cached slots 0..P-1, then its own (bf16-rounded)
            att = []
            for j in range(nq):
                hk = j // group
                keys = [[_bf(x) for x in kv[l, 0, b, hk, t]] for t in range(P)]
                vals = [[_bf(x) for x in kv[l, 1, b, hk, t]] for t in range(P)]
                keys.append([float(numerics.round_to_bf16(np.array(x))) for x in kh[hk]])
                vals.append([float(numerics.round_to_bf16(np.array(x))) for x in vh[hk]])
                if kv_out is not None and j % group == 0:
                    kv_out[l, 0, b, hk, P] = numerics.f64_to_bf16_bits(np.array(kh[hk]))
                    kv_out[l, 1, b, hk, P] = numerics.f64_to_bf16_bits(np.array(vh[hk]))
                sc = [sum(qh[j][i] * key[i] for i in range(d)) / math.sqrt(d) for key in keys]
                mx = max(sc)
                ex = [math.exp(s - mx) for s in sc]
                tot = sum(ex)
                att.extend(sum(ex[t] / tot * vals[t][i] for t in range(P + 1)) for i in range(d))
            o = matvec(lay["o"], att, H)
            h = [h[i] + o[i] for i in range(H)]
            xn = norm(h, lay["post_norm"])
            gt = matvec(lay["gate"], xn, I)
            up = matvec(lay["up"], xn, I)
            g = [gt[i] / (1.0 + math.exp(-gt[i])) * up[i] for i in range(I)]
            dn = matvec(lay["down"], g, H)
            h = [h[i] + dn[i] for i in range(H)]
        out_logits.append(matvec(model["lm_head"], norm(h, model["final_norm"]), V))
    return np.array(out_logits)


def _np_model(model):
    def conv(x):
        if isinstance(x, dict):
            return {k: conv(v) for k, v in x.items()}
        if isinstance(x, list):
            return [conv(v) for v in x]
        return oracle.decoder._to_numpy(x)
    return {k: conv(v) for k, v in model.items()}


@pytest.mark.parametrize("fmt", [synthetic.BF16, synthetic.AFFINE4_G64])
def test_step_matches_scalar_restatement(fmt):
    wl = synthetic.custom(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
                          intermediate=128, vocab=40, weight_format=fmt, batch=2, prefill=5, steps=1,
                          seed=7)
    model = synthetic.generate(wl)
    model["positions"][1] = 2  # ragged lengths
    npm = _np_model(model)
    kv = npm["kv"].copy()
    m = oracle.OracleModel.from_synthetic(wl, model)
    logits, am = oracle.decode_step(m, kv, npm["tokens"], npm["positions"])
    ref = _scalar_step(wl, npm, npm["kv"], npm["tokens"], npm["positions"])
    assert np.allclose(logits, ref, rtol=1e-11, atol=1e-12)
    assert am.tolist() == [int(np.argmax(r)) for r in ref]


def test_step_writes_only_slot_p_and_ignores_later_slots():
    wl = synthetic.custom(n_layers=2, hidden=64, n_q_heads=2, n_kv_heads=1, head_dim=32, intermediate=96,
                          vocab=50, batch=2, prefill=6, steps=3, seed=3)
    model = synthetic.generate(wl)
    npm = _np_model(model)
    P = npm["positions"]
    kv0 = npm["kv"].copy()
    kv = kv0.copy()
    m = oracle.OracleModel.from_synthetic(wl, model)
    logits, _ = oracle.decode_step(m, kv, npm["tokens"], P)
    changed = np.argwhere(kv != kv0)
    assert len(changed) > 0
    for l, p, b, h, t, i in changed:
        assert t == P[b]
    # junk in the slots after P must not change anything
    kv_junk = kv0.copy()
    for b in range(2):
        kv_junk[:, :, b, :, P[b] + 1:, :] = numerics.f64_to_bf16_bits(np.full_like(
            kv_junk[:, :, b, :, P[b] + 1:, :], 1000.0, dtype=np.float64))
    logits2, _ = oracle.decode_step(m, kv_junk, npm["tokens"], P)
    assert np.array_equal(logits, logits2)


def test_step_sequences_are_independent():
    wl = synthetic.custom(n_layers=1, hidden=64, n_q_heads=2, n_kv_heads=1, head_dim=32, intermediate=96,
                          vocab=50, batch=3, prefill=4, steps=1, seed=11)
    model = synthetic.generate(wl)
    npm = _np_model(model)
    npm["positions"][:] = [4, 1, 3]
    m = oracle.OracleModel.from_synthetic(wl, model)
    kv = npm["kv"].copy()
    logits, am = oracle.decode_step(m, kv, npm["tokens"], npm["positions"])
    for b in range(3):
        wl1 = wl.replace(batch=1)
        m1 = oracle.OracleModel(wl1, m.raw)
        kv1 = npm["kv"][:, :, b:b + 1].copy()
        l1, a1 = oracle.decode_step(m1, kv1, npm["tokens"][b:b + 1], npm["positions"][b:b + 1])
        assert np.allclose(l1[0], logits[b], rtol=1e-13, atol=1e-13)
        assert np.array_equal(kv1[:, :, 0], kv[:, :, b])


def _verify_case(fmt=synthetic.BF16):
    wl = synthetic.custom(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, intermediate=128,
                          vocab=40, weight_format=fmt, batch=2, prefill=5, steps=4, seed=21)
    model = synthetic.generate(wl)
    model["positions"][1] = 2  # ragged lengths
    npm = _np_model(model)
    rng = np.random.default_rng(5)
    toks = rng.integers(0, wl.vocab, (2, 3)).astype(np.int32)
    return wl, model, npm, toks


@pytest.mark.parametrize("fmt", [synthetic.BF16, synthetic.AFFINE4_G64])
def test_verify_step_matches_scalar_teacher_forcing(fmt):
    """Row (b, t) of the verify step is the one-token step of sequence b at position P_b + t
    after rows (b, 0..t-1) were appended: the scalar restatement, run row by row and
    writing each row's K/V into its own cache copy, gives the same logits and cache."""
    wl, model, npm, toks = _verify_case(fmt)
    m = oracle.OracleModel.from_synthetic(wl, model)
    kv = npm["kv"].copy()
    logits, am = oracle.verify_step(m, kv, toks, npm["positions"])
    assert logits.shape == (2, 3, wl.vocab) and am.shape == (2, 3)
    kv_s = npm["kv"].copy()
    for t in range(3):
        ref = _scalar_step(wl, npm, kv_s, toks[:, t], npm["positions"] + t, kv_out=kv_s)
        assert np.allclose(logits[:, t], ref, rtol=1e-11, atol=1e-12), f"row {t}"
        assert am[:, t].tolist() == [int(np.argmax(r)) for r in ref]
    assert np.array_equal(kv, kv_s)
    # slots P_b .. P_b + 2 written, nothing else
    changed = np.argwhere(np.any(kv != npm["kv"], axis=-1))
    for l, p, b, h, slot in changed:
        assert npm["positions"][b] <= slot < npm["positions"][b] + 3


def test_verify_step_rows_do_not_see_later_tokens():
    """Causality inside the step: row t does not depend on the tokens of rows t+1 .. T-1."""
    wl, model, npm, toks = _verify_case()
    m = oracle.OracleModel.from_synthetic(wl, model)
    lg1, _ = oracle.verify_step(m, npm["kv"].copy(), toks, npm["positions"])
    toks2 = toks.copy()
    toks2[:, 2] = (toks2[:, 2] + 7) % wl.vocab
    lg2, _ = oracle.verify_step(m, npm["kv"].copy(), toks2, npm["positions"])
    assert np.array_equal(lg1[:, :2], lg2[:, :2])
    assert not np.allclose(lg1[:, 2], lg2[:, 2])


def test_verify_step_of_one_token_is_the_decode_step():
    wl, model, npm, toks = _verify_case()
    m = oracle.OracleModel.from_synthetic(wl, model)
    kv1, kv2 = npm["kv"].copy(), npm["kv"].copy()
    lg, am = oracle.verify_step(m, kv1, toks[:, :1], npm["positions"])
    ref = _scalar_step(wl, npm, npm["kv"], toks[:, 0], npm["positions"], kv_out=kv2)
    assert np.allclose(lg[:, 0], ref, rtol=1e-11, atol=1e-12)
    assert np.array_equal(kv1, kv2)

"""Pins for the oracle's affine 8-bit KV cache format (oracle/kvcache.py): hand-worked
groups, brute-force optimality of every code, ends and monotonicity of the decode,
the error bound, and a decode step over a quantized cache against a scalar-loop
restatement (its own quantizer, written with Python floats and float32 scalars)."""

import math
import pathlib

import numpy as np
import pytest

import oracle
import synthetic
from oracle import kvcache, numerics

GOLDEN = pathlib.Path(__file__).parent / "golden"
rng = np.random.default_rng(77)


def _cases():
    out = []
    for line in (GOLDEN / "affine8_kv_worked_examples.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        name, fill, vals, sb, codes, fill_code = [f.strip() for f in line.split("|")]
        x = np.full(64, float(fill))
        for kv in vals.split():
            i, v = kv.split("=")
            x[int(i)] = float(v)
        want = np.full(64, int(fill_code))
        for kv in codes.split():
            i, c = kv.split("=")
            want[int(i)] = int(c)
        s, b = (float(v) for v in sb.split())
        out.append(pytest.param(x, s, b, want, id=name))
    return out


@pytest.mark.parametrize("x,scale,bias,codes", _cases())
def test_hand_worked_groups(x, scale, bias, codes):
    c, s, b = oracle.quantize_affine8_g64(x[None, :])
    assert numerics.bf16_bits_to_f64(s).item() == scale
    assert numerics.bf16_bits_to_f64(b).item() == bias
    assert c[0].tolist() == codes.tolist()


def _random_groups(n):
    """Rows of 64 with random location and spread (bf16 range, float32 values)."""
    loc = rng.standard_normal((n, 1)) * 3
    spread = np.exp(rng.uniform(-6, 3, (n, 1)))
    return (loc + spread * rng.standard_normal((n, 64))).astype(np.float32)


def test_every_code_is_the_nearest_level():
    # brute force over all 256 levels in float64: the chosen code is a nearest level of
    # scale * c + bias to x (float32 decisions can only differ on a near tie)
    x = _random_groups(300)
    c, sb, bb = oracle.quantize_affine8_g64(x)
    s = numerics.bf16_bits_to_f64(sb)[:, :1]
    b = numerics.bf16_bits_to_f64(bb)[:, :1]
    levels = s[:, :, None] * np.arange(256)[None, None, :] + b[:, :, None]  # [n, 1, 256]
    dist = np.abs(levels - x.astype(np.float64)[:, :, None])                # [n, 64, 256]
    best = dist.min(axis=-1)
    chosen = np.take_along_axis(dist, c[:, :, None].astype(np.int64), axis=-1)[..., 0]
    tie_slack = 1e-5 * s + 1e-12
    assert np.all(chosen <= best + tie_slack)


def test_decode_ends_monotonicity_and_bound():
    x = _random_groups(200)
    c, sb, bb = oracle.quantize_affine8_g64(x)
    y = oracle.dequant_affine8_g64(c, sb, bb)
    s = numerics.bf16_bits_to_f64(sb)
    b = numerics.bf16_bits_to_f64(bb)
    # code 0 reads the bias, code 255 reads bias + 255 scale, exactly
    assert np.array_equal(oracle.dequant_affine8_g64(np.zeros_like(c), sb, bb), np.repeat(b, 64, axis=1))
    assert np.array_equal(oracle.dequant_affine8_g64(np.full_like(c, 255), sb, bb), np.repeat(b + 255 * s, 64, axis=1))
    # order is kept within a group
    for r in range(x.shape[0]):
        o = np.argsort(x[r], kind="stable")
        assert np.all(np.diff(c[r][o].astype(int)) >= 0)
    # |x - read| <= half a level, plus what the bf16 rounding of bias and scale moved the ends
    mn, mx = x.min(axis=1, keepdims=True).astype(np.float64), x.max(axis=1, keepdims=True).astype(np.float64)
    ends = np.maximum(np.abs(b - mn), np.abs(b + 255 * s - mx))
    err = np.abs(y - x.astype(np.float64))
    assert np.all(err <= s / 2 + ends + 1e-6 * (np.abs(mx) + np.abs(mn)))


def test_groups_are_independent_and_rows_of_two_groups():
    x = _random_groups(4).reshape(2, 128)
    c, sb, bb = oracle.quantize_affine8_g64(x)
    for g in range(2):
        c1, s1, b1 = oracle.quantize_affine8_g64(x[:, 64 * g:64 * (g + 1)])
        assert np.array_equal(c[:, 64 * g:64 * (g + 1)], c1)
        assert np.array_equal(sb[:, g:g + 1], s1) and np.array_equal(bb[:, g:g + 1], b1)


def test_float64_input_is_taken_to_float32_first():
    x64 = rng.standard_normal((8, 64))
    a = oracle.quantize_affine8_g64(x64)
    b = oracle.quantize_affine8_g64(x64.astype(np.float32))
    assert all(np.array_equal(u, v) for u, v in zip(a, b))


# ------------------------------------------------------------- a step over a quantized cache

def _bf(bits):
    return float(numerics.bf16_bits_to_f64(np.array([bits], dtype=np.uint16))[0])


def _scalar_quant(row):
    """Min-max affine 8-bit quantization of one group, restated with float32 scalars."""
    f = np.float32
    xs = [f(v) for v in row]
    mn, mx = min(xs), max(xs)
    scale = float(numerics.round_to_bf16(np.array(float(f(f(mx - mn) / f(255.0))))))
    bias = float(numerics.round_to_bf16(np.array(float(mn))))
    out = []
    for v in xs:
        if scale == 0.0:
            out.append(bias)
            continue
        t = float(f(f(v - f(bias)) / f(scale)))
        code = min(255.0, max(0.0, float(np.rint(t))))
        out.append(scale * code + bias)
    return out


def _scalar_step_kv8(wl, npm, tokens, positions):
    """The decode step with Python scalars, reading the quantized cache element by element
    and quantizing the new row with _scalar_quant (shared helper: bf16 reading only)."""
    L, H, nq, nkv, d, I, V = (wl.n_layers, wl.hidden, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                              wl.intermediate, wl.vocab)
    eps, theta, group = wl.rms_eps, wl.rope_theta, nq // nkv
    codes, params = npm["kv"]["codes"], npm["kv"]["params"]

    def mv(w, x, n):
        return [sum(_bf(w[r, c]) * x[c] for c in range(len(x))) for r in range(n)]

    def norm(x, w):
        inv = 1.0 / math.sqrt(sum(v * v for v in x) / len(x) + eps)
        return [x[i] * inv * _bf(w[i]) for i in range(len(x))]

    def rope(x, pos):
        half, y = d // 2, [0.0] * d
        for i in range(half):
            a = pos * theta ** (-2.0 * i / d)
            y[i] = x[i] * math.cos(a) - x[i + half] * math.sin(a)
            y[i + half] = x[i + half] * math.cos(a) + x[i] * math.sin(a)
        return y

    def cached(l, p, b, h, t):
        return [_bf(params[l, p, b, h, t, i // 64, 0]) * float(codes[l, p, b, h, t, i])
                + _bf(params[l, p, b, h, t, i // 64, 1]) for i in range(d)]

    out = []
    for b in range(len(tokens)):
        P = int(positions[b])
        h = [_bf(v) for v in npm["embed"][int(tokens[b])]]
        for l in range(L):
            lay = npm["layers"][l]
            xn = norm(h, lay["in_norm"])
            q, k, v = mv(lay["q"], xn, nq * d), mv(lay["k"], xn, nkv * d), mv(lay["v"], xn, nkv * d)
            qh = [rope(norm(q[j * d:(j + 1) * d], lay["q_norm"]), P) for j in range(nq)]
            kh = [rope(norm(k[j * d:(j + 1) * d], lay["k_norm"]), P) for j in range(nkv)]
            att = []
            for j in range(nq):
                hk = j // group
                keys = [cached(l, 0, b, hk, t) for t in range(P)] + [
                    sum((_scalar_quant(kh[hk][g:g + 64]) for g in range(0, d, 64)), [])]
                vals = [cached(l, 1, b, hk, t) for t in range(P)] + [
                    sum((_scalar_quant(v[hk * d + g:hk * d + g + 64]) for g in range(0, d, 64)), [])]
                sc = [sum(qh[j][i] * key[i] for i in range(d)) / math.sqrt(d) for key in keys]
                mx = max(sc)
                ex = [math.exp(s - mx) for s in sc]
                tot = sum(ex)
                att.extend(sum(ex[t] / tot * vals[t][i] for t in range(P + 1)) for i in range(d))
            h = [h[i] + o for i, o in enumerate(mv(lay["o"], att, H))]
            xn = norm(h, lay["post_norm"])
            gt, up = mv(lay["gate"], xn, I), mv(lay["up"], xn, I)
            g = [gt[i] / (1.0 + math.exp(-gt[i])) * up[i] for i in range(I)]
            h = [h[i] + o for i, o in enumerate(mv(lay["down"], g, H))]
        out.append(mv(npm["lm_head"], norm(h, npm["final_norm"]), V))
    return np.array(out)


def _kv8_model(seed=5, head_dim=64, batch=2, prefill=4, **kw):
    wl = synthetic.custom(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=head_dim,
                          intermediate=96, vocab=40, batch=batch, prefill=prefill, steps=2, seed=seed,
                          kv_format=synthetic.AFFINE8_G64, **kw)
    model = synthetic.generate(wl)
    from tests.parity import np_model
    return wl, model, np_model(model)


def _cache(npm):
    return oracle.Affine8Cache(npm["kv"]["codes"].copy(), npm["kv"]["params"].copy())


@pytest.mark.parametrize("head_dim", [64, 128])
def test_kv8_step_matches_scalar_restatement(head_dim):
    wl, model, npm = _kv8_model(head_dim=head_dim)
    npm["positions"][1] = 1  # ragged
    m = oracle.OracleModel.from_synthetic(wl, model)
    kv = _cache(npm)
    logits, am = oracle.decode_step(m, kv, npm["tokens"], npm["positions"])
    ref = _scalar_step_kv8(wl, npm, npm["tokens"], npm["positions"])
    assert np.allclose(logits, ref, rtol=1e-10, atol=1e-11)
    assert am.tolist() == [int(np.argmax(r)) for r in ref]


def test_kv8_step_writes_slot_p_in_the_stored_form():
    wl, model, npm = _kv8_model(seed=9)
    m = oracle.OracleModel.from_synthetic(wl, model)
    kv0 = _cache(npm)
    kv = kv0.copy()
    oracle.decode_step(m, kv, npm["tokens"], npm["positions"])
    P = npm["positions"]
    ch = np.argwhere(kv.codes != kv0.codes)
    assert len(ch) > 0 and all(t == P[b] for _, _, b, _, t, _ in ch)
    chp = np.argwhere(kv.params != kv0.params)
    assert len(chp) > 0 and all(t == P[b] for _, _, b, _, t, _, _ in chp)
    # each written row is a valid quantization: its own min and max land on codes 0 / near 255
    for l in range(wl.n_layers):
        for p in range(2):
            c = kv.codes[l, p, 0, :, P[0]]
            assert c.min() == 0 and c.max() >= 250

"""Pins for the CPU oracle: closed forms, special cases, invariants and brute
force that hold independently of the oracle's own code.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong pairing) fails it.
"""

import math
import pathlib

import numpy as np
import pytest
import torch

import oracle
from oracle import affine4, numerics
from oracle.decoder import attention_partial

GOLDEN = pathlib.Path(__file__).parent / "golden"
rng = np.random.default_rng(1234)


# ------------------------------------------------------------------ bf16

def test_bf16_read_exact():
    # 0x3F80 = 1.0, 0xC000 = -2.0, 0x3F81 = 1 + 2^-7, 0x0000 = 0
    got = numerics.bf16_bits_to_f64(np.array([0x3F80, 0xC000, 0x3F81, 0x0000], dtype=np.uint16))
    assert got.tolist() == [1.0, -2.0, 1.0 + 2.0 ** -7, 0.0]


def test_bf16_round_half_even_cases():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: goes to 1 + 2^-6 (0x3F82)
    # 1 + 2^-8 + 2^-30 is just above halfway: rounds up to 0x3F81
    xs = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -30, -(1 + 2.0 ** -8)])
    assert numerics.f64_to_bf16_bits(xs).tolist() == [0x3F80, 0x3F82, 0x3F81, 0xBF80]


def test_bf16_round_matches_torch_on_float32_inputs():
    # float32 inputs: a single rounding to bf16, the same in both (library routine)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ours = numerics.f64_to_bf16_bits(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------------ affine 4-bit

def _golden_affine():
    rows = []
    for line in (GOLDEN / "affine4_worked_examples.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        lhs, rhs = line.split("->")
        word, scale, bias = lhs.split()
        rows.append((int(word, 16), float(scale), float(bias), [float(v) for v in rhs.split()]))
    return rows


@pytest.mark.parametrize("word,scale,bias,expect", _golden_affine())
def test_dequant_hand_worked(word, scale, bias, expect):
    # one row of 64 inputs = 8 words; put the example word first, zeros after
    words = np.zeros((1, 8), dtype=np.uint32)
    words[0, 0] = word
    s = numerics.f64_to_bf16_bits(np.array([[scale]]))
    b = numerics.f64_to_bf16_bits(np.array([[bias]]))
    w = affine4.dequant_affine4_g64(words, s, b)
    assert w.shape == (1, 64)
    assert w[0, :8].tolist() == expect
    assert np.all(w[0, 8:] == bias)


def test_dequant_groups_and_rows_are_independent():
    # 2 rows x 128 inputs (2 groups): each (row, group) uses its own scale/bias
    words = np.full((2, 16), 0x76543210, dtype=np.uint32)
    scales = np.array([[1.0, 2.0], [4.0, 8.0]])
    biases = np.array([[0.0, 1.0], [-1.0, 0.5]])
    w = affine4.dequant_affine4_g64(words, numerics.f64_to_bf16_bits(scales), numerics.f64_to_bf16_bits(biases))
    q = np.tile(np.arange(8), 16)
    for r in range(2):
        for g in range(2):
            np.testing.assert_array_equal(w[r, 64 * g:64 * (g + 1)], scales[r, g] * q[:64] + biases[r, g])


def test_dequant_unit_scale_gives_integers():
    words = rng.integers(0, 2 ** 32, size=(3, 16), dtype=np.uint64).astype(np.uint32)
    one = numerics.f64_to_bf16_bits(np.ones((3, 2)))
    zero = numerics.f64_to_bf16_bits(np.zeros((3, 2)))
    w = affine4.dequant_affine4_g64(words, one, zero)
    # brute force: nibble k of word j, by string formatting of the hex digits
    for r in range(3):
        for j in range(16):
            hexdigits = f"{int(words[r, j]):08x}"[::-1]  # lowest nibble first
            assert [int(c, 16) for c in hexdigits] == w[r, 8 * j:8 * j + 8].astype(int).tolist()


def test_affine_offset_rewrite_identity():
    # oxinfer "MLX checkpoints": scale*q + bias == scale*(q-8) + (bias + 8*scale)
    s = numerics.round_to_bf16(rng.uniform(0.001, 0.01, 1000))
    b = numerics.round_to_bf16(rng.normal(0, 0.02, 1000))
    q = rng.integers(0, 16, 1000).astype(np.float64)
    assert np.array_equal(s * q + b, s * (q - 8) + (b + 8 * s))


def test_dequant_f32_is_single_rounding():
    words = rng.integers(0, 2 ** 32, size=(4, 32), dtype=np.uint64).astype(np.uint32)
    s = numerics.f64_to_bf16_bits(rng.uniform(0.001, 0.01, (4, 4)))
    b = numerics.f64_to_bf16_bits(rng.normal(0, 0.02, (4, 4)))
    w64 = affine4.dequant_affine4_g64(words, s, b)
    w32 = affine4.dequant_affine4_g64_f32(words, s, b)
    # the float32 value is the nearest float32 to the exact float64 value
    err = np.abs(w32.astype(np.float64) - w64)
    ulp = np.spacing(np.abs(w32)).astype(np.float64)
    assert np.all(err <= 0.5 * ulp)


# ------------------------------------------------------------------ RMSNorm / SiLU / softmax / argmax

def test_rmsnorm_hand_value_and_unit_rms():
    y = oracle.rmsnorm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    # mean(x^2) = 12.5
    assert np.allclose(y, [3 / math.sqrt(12.5), 8 / math.sqrt(12.5)], rtol=0, atol=1e-15)
    x = rng.standard_normal(256)
    y = oracle.rmsnorm(x, np.ones(256), 1e-6)
    ms = np.mean(x * x)
    assert abs(np.sqrt(np.mean(y * y)) - np.sqrt(ms / (ms + 1e-6))) < 1e-14


def test_rmsnorm_scale_invariant_without_eps():
    x = rng.standard_normal(64)
    w = rng.standard_normal(64)
    assert np.allclose(oracle.rmsnorm(x, w, 0.0), oracle.rmsnorm(7.5 * x, w, 0.0), rtol=1e-14, atol=0)


def test_silu_special_values():
    assert oracle.silu(np.array(0.0)) == 0.0
    assert abs(float(oracle.silu(np.array(1.0))) - 0.7310585786300049) < 1e-15  # 1/(1+e^-1)
    assert abs(float(oracle.silu(np.array(40.0))) - 40.0) < 1e-12
    assert abs(float(oracle.silu(np.array(-40.0)))) < 1e-15


def test_softmax_rows_sum_to_one():
    s = rng.standard_normal((50, 300)) * 10
    p = oracle.softmax(s)
    assert np.all(np.abs(p.sum(-1) - 1) < 1e-12)
    assert np.all(p > 0)


def test_argmax_lowest_index_on_ties():
    assert oracle.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert oracle.argmax_lowest(np.array([5.0, 5.0])) == 0
    assert oracle.argmax_lowest(np.array([-1.0, -0.5, -2.0])) == 1


def test_tie_exemption_threshold():
    assert oracle.tie_exempt(np.array([10.0, 9.95, 0.0]))        # gap 0.05 < 0.1
    assert not oracle.tie_exempt(np.array([10.0, 9.8, 0.0]))     # gap 0.2 >= 0.1


# ------------------------------------------------------------------ RoPE

def test_rope_identity_at_position_zero():
    x = rng.standard_normal((3, 128))
    assert np.array_equal(oracle.rope_rotate_half(x, 0, 1e6), x)


def test_rope_rotate_half_pairing_and_frequency():
    # d = 4, theta = 1e6: angles are pos * 1e6^0 = pos and pos * 1e6^(-1/2) = pos/1000
    e0 = np.array([1.0, 0, 0, 0])
    y = oracle.rope_rotate_half(e0, 1, 1e6)
    # element 0 pairs with element 2 (i with i + d/2), rotating by angle 1
    assert np.allclose(y, [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    e1 = np.array([0, 1.0, 0, 0])
    y = oracle.rope_rotate_half(e1, 5, 1e6)
    assert np.allclose(y, [0, math.cos(0.005), 0, math.sin(0.005)], atol=1e-15)
    e2 = np.array([0, 0, 1.0, 0])
    y = oracle.rope_rotate_half(e2, 1, 1e6)
    assert np.allclose(y, [-math.sin(1), 0, math.cos(1), 0], atol=1e-15)


def test_rope_preserves_pair_norms():
    x = rng.standard_normal(128)
    y = oracle.rope_rotate_half(x, 777, 1e6)
    n_x = x[:64] ** 2 + x[64:] ** 2
    n_y = y[:64] ** 2 + y[64:] ** 2
    assert np.allclose(n_x, n_y, rtol=1e-13, atol=0)


def test_rope_scores_depend_only_on_relative_position():
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    a = oracle.rope_rotate_half(q, 1000, 1e6) @ oracle.rope_rotate_half(k, 990, 1e6)
    b = oracle.rope_rotate_half(q, 5010, 1e6) @ oracle.rope_rotate_half(k, 5000, 1e6)
    assert abs(a - b) < 1e-9


# ------------------------------------------------------------------ attention

def test_attention_single_key_returns_its_value():
    q = rng.standard_normal((4, 64))
    K = rng.standard_normal((2, 1, 64))
    V = rng.standard_normal((2, 1, 64))
    o = oracle.gqa_attention(q, K, V)
    # query heads 0,1 share kv head 0; heads 2,3 share kv head 1 (j // group)
    assert np.array_equal(o, np.stack([V[0, 0], V[0, 0], V[1, 0], V[1, 0]]))


def test_attention_identical_keys_average_values():
    q = rng.standard_normal((2, 64))
    k = rng.standard_normal(64)
    K = np.tile(k, (1, 9, 1))
    V = rng.standard_normal((1, 9, 64))
    o = oracle.gqa_attention(q, K, V)
    assert np.allclose(o, np.tile(V[0].mean(0), (2, 1)), rtol=0, atol=1e-14)


def test_attention_scale_is_inverse_sqrt_head_dim():
    d = 16
    # two keys whose scores differ by sqrt(d) * ln 3 before scaling -> weights 3/4, 1/4
    q = np.zeros((1, d)); q[0, 0] = 1.0
    K = np.zeros((1, 2, d)); K[0, 0, 0] = math.sqrt(d) * math.log(3.0)
    V = np.zeros((1, 2, d)); V[0, 0, 1] = 1.0; V[0, 1, 2] = 1.0
    o = oracle.gqa_attention(q, K, V)
    assert np.allclose(o[0, 1:3], [0.75, 0.25], atol=1e-15)


def test_lse_merge_of_any_partition_equals_one_pass():
    q = rng.standard_normal(128)
    K = rng.standard_normal((1000, 128)) * 2
    V = rng.standard_normal((1000, 128))
    ref = oracle.gqa_attention(q[None], K[None], V[None])[0]
    for cuts in ([0, 1000], [0, 1, 1000], [0, 333, 334, 999, 1000], list(range(0, 1001, 64)) + [1000]):
        cuts = sorted(set(cuts))
        parts = [attention_partial(q, K[a:b], V[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
        assert np.allclose(oracle.lse_merge(parts), ref, rtol=0, atol=1e-13)


# ------------------------------------------------------------------ GEMV brute force

def test_linear_matches_nested_loops_on_small_integers():
    from synthetic import custom
    wl = custom(hidden=64, intermediate=128, vocab=96, n_q_heads=2, n_kv_heads=1, head_dim=32)
    W = rng.integers(-8, 8, size=(96, 64)).astype(np.float64)     # non-square: catches a transpose
    bits = numerics.f64_to_bf16_bits(W)
    m = oracle.OracleModel(wl, {"lm_head": bits})
    x = rng.integers(-5, 6, size=(3, 64)).astype(np.float64)
    y = m.linear(x, "lm_head")
    for b in range(3):
        for r in range(96):
            acc = 0.0
            for c in range(64):
                acc += W[r, c] * x[b, c]
            assert y[b, r] == acc

"""The GPU tests' comparison helpers, exercised on the CPU with mistakes planted in oracle
results (no GPU): the tolerance rule rejects any sequence outside max|dlogit| <= 5e-2 or
rel L2 <= 1e-2 and any argmax mismatch outside the top-2 near-tie margin; a replay of a
subset of a batch gives exactly the full replay's rows for those sequences."""

import numpy as np
import pytest

import oracle
import synthetic
from parity import MAX_ABS, REL_L2, check_logits, np_model, oracle_replay, replay_plan


def _tiny(kv_format=synthetic.BF16, batch=3):
    wl = synthetic.custom(name="helpers", seed=4, n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=64,
                          intermediate=128, vocab=50, batch=batch, prefill=(3, 9), steps=3, kv_format=kv_format)
    model = synthetic.generate(wl)
    npm = np_model(model)
    if kv_format == synthetic.BF16:
        kv = npm["kv"]
    else:
        kv = oracle.Affine8Cache(npm["kv"]["codes"].copy(), npm["kv"]["params"].copy())
    return wl, model, npm, kv


def test_planted_mistakes_are_rejected():
    wl, model, npm, kv = _tiny()
    m = oracle.OracleModel.from_synthetic(wl, model)
    ref, am = oracle.decode_step(m, kv.copy(), npm["tokens"], npm["positions"])
    w = check_logits(ref.copy(), ref, am, am, "same")
    assert w["max_abs"] == 0.0 and w["exempt"] == 0
    bad = ref.copy()
    bad[1, 7] += 1.5 * MAX_ABS  # one logit of sequence 1 beyond the absolute tolerance
    with pytest.raises(AssertionError, match="seq 1: max"):
        check_logits(bad, ref, am, am, "planted")
    bad = ref * (1 + 2 * REL_L2)  # every logit of every sequence 2% off: beyond rel L2
    with pytest.raises(AssertionError, match="seq 0"):
        check_logits(bad, ref, am, am, "planted")
    wrong = am.copy()
    wrong[2] = (am[2] + 1) % wl.vocab  # an argmax that is not a near tie
    assert not oracle.tie_exempt(ref[2])
    with pytest.raises(AssertionError, match="outside the tie margin"):
        check_logits(ref, ref, wrong, am, "planted")


def test_near_tie_is_the_only_argmax_exemption():
    ref = np.linspace(-3.0, 2.0, 40)[None, :].copy()
    ref[0, 10] = 2.0 - 0.5e-2 * 3.0  # second best within 1e-2 * max|logit| (3.0) of the best
    am = np.array([39])
    w = check_logits(ref.copy(), ref, np.array([10]), am, "tie")
    assert w["exempt"] == 1
    ref[0, 10] = 2.0 - 2e-2 * 3.0  # outside the margin
    with pytest.raises(AssertionError, match="outside the tie margin"):
        check_logits(ref.copy(), ref, np.array([10]), am, "no tie")


@pytest.mark.parametrize("fmt", [synthetic.BF16, synthetic.AFFINE8_G64])
def test_subset_replay_equals_the_full_replay(fmt):
    """oracle_replay over sequences (0, 2) of a batch of 3 gives the full replay's logits,
    argmax and cache of those sequences (the sequences of a batch are independent)."""
    wl, model, npm, kv = _tiny(fmt)
    m = oracle.OracleModel.from_synthetic(wl, model)
    # a greedy token sequence from the oracle itself stands in for the GPU's
    steps = []
    tok, pos, k = npm["tokens"].copy(), npm["positions"].copy(), kv.copy()
    for _ in range(wl.steps):
        lg, a = oracle.decode_step(m, k, tok, pos)
        steps.append((tok.copy(), pos.copy(), lg, a))
        tok, pos = a.astype(np.int32), pos + 1
    full, kv_full = oracle_replay(wl, model, kv, steps, model=m)
    sub, kv_sub = oracle_replay(wl, model, kv, steps, seqs=[0, 2], model=m)
    for (s1, l1, a1), (s2, l2, a2) in zip(full, sub):
        assert s1 == s2
        assert np.array_equal(l1[[0, 2]], l2) and np.array_equal(a1[[0, 2]], a2)
    if fmt == synthetic.BF16:
        assert np.array_equal(kv_full[:, :, [0, 2]], kv_sub)
    else:
        assert np.array_equal(kv_full.codes[:, :, [0, 2]], kv_sub.codes)
        assert np.array_equal(kv_full.params[:, :, [0, 2]], kv_sub.params)


def test_replay_plan_covers_every_step():
    for name, wl in synthetic.WORKLOADS.items():
        plan = replay_plan(wl)
        assert any(n == wl.steps for _, n in plan), name
        assert any(seqs is None for seqs, _ in plan), name  # every sequence is checked at some step
        if wl.batch > 4:
            seqs = next(s for s, n in plan if n == wl.steps)
            assert 0 in seqs and wl.batch - 1 in seqs

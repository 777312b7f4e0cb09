"""The GPU tests' comparison helpers, exercised on the CPU with mistakes planted in oracle
results: the conditioning check must reject a wrong result on a well-conditioned model and
may only exempt a sequence whose oracle answer itself moves beyond the tolerance."""

import numpy as np
import pytest

import oracle
import synthetic
from parity import MAX_ABS, check_logits_conditioned, np_model, oracle_noise_spread


def _tiny(kv_format=synthetic.BF16):
    wl = synthetic.custom(name="cond", seed=4, n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=64,
                          intermediate=128, vocab=50, batch=2, prefill=8, steps=2, kv_format=kv_format)
    model = synthetic.generate(wl)
    npm = np_model(model)
    if kv_format == synthetic.BF16:
        kv = npm["kv"]
    else:
        kv = oracle.Affine8Cache(npm["kv"]["codes"].copy(), npm["kv"]["params"].copy())
    return wl, model, npm, kv


@pytest.mark.parametrize("fmt", [synthetic.BF16, synthetic.AFFINE8_G64])
def test_spread_of_a_well_conditioned_model_is_small(fmt):
    wl, model, npm, kv = _tiny(fmt)
    steps = [(npm["tokens"], npm["positions"], None, None)]
    spread = oracle_noise_spread(wl, model, kv, steps, 0, 1, cache_weights=True)
    assert 0.0 < spread < 1e-3


def test_planted_mistake_is_rejected_and_exemption_needs_spread():
    wl, model, npm, kv = _tiny()
    m = oracle.OracleModel.from_synthetic(wl, model)
    ref, am = oracle.decode_step(m, kv.copy(), npm["tokens"], npm["positions"])
    bad = ref.copy()
    bad[1] += 0.5  # a wrong result for sequence 1
    with pytest.raises(AssertionError, match="seq 1"):
        check_logits_conditioned(bad, ref, am, am, "planted", lambda b: 1e-6)
    # only when the oracle's own spread exceeds the tolerance is the sequence exempted
    w = check_logits_conditioned(bad, ref, am, am, "planted", lambda b: 10 * MAX_ABS)
    assert w["ill_conditioned"] == 1
    # a correct result passes without calling the check
    w = check_logits_conditioned(ref, ref, am, am, "same", lambda b: pytest.fail("not needed"))
    assert w["ill_conditioned"] == 0 and w["max_abs"] == 0.0

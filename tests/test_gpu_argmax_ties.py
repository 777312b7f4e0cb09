"""Exact argmax ties on the GPU: every lm_head epilogue (the batch-1 GEMV, the batched
projections on mma.sync and on tcgen05, the tensor-memory prefill projections) must return
the lowest index among equal maxima, also when the equal logits sit in different vocab tiles
and different CTAs, and must agree with its own logits output (argmax = first index of the
row's maximum).

Ties are built, not hoped for: (1) an all-zero lm_head makes every logit +0, so the whole
vocabulary ties and the answer is index 0; (2) the lm_head row that won a first step is
copied to rows 256, 512, ... above and below it (the same position inside every tile of 8, 16, 128
or 256 rows, so the copies take the same arithmetic and their logits are bit-identical,
which the test checks; for the stream-K tcgen05 kernel, whose tiles are split at differing
K offsets, to other warps and lanes of the winner's own tile) and the step is run again on
the same inputs.
Sources: Butter architecture.md, GPU sampling section (greedy = argmax over the vocab);
ANEForge "LLMs on the ANE", "lm_head on the ANE" (the vocab split into tiles, each with
its own maximum)."""

import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu

# name, weight format, batch, tokens per sequence, hidden: which lm_head epilogue runs (the
# tc_decode cases select the tcgen05 decode projections, dec_config.proj_kernels = 2)
CASES = [
    ("gemv_bf16", synthetic.BF16, 1, 1, 256),
    ("gemv_q4", synthetic.AFFINE4_G64, 1, 1, 256),
    ("batched_bf16_b5", synthetic.BF16, 5, 1, 256),
    ("batched_q4_b12", synthetic.AFFINE4_G64, 12, 1, 256),
    ("batched_q4_b32", synthetic.AFFINE4_G64, 32, 1, 512),
    ("prefill_tc_bf16_t128", synthetic.BF16, 1, 128, 2048),
    # hidden >= 2048 at 2..32 rows: the tcgen05 decode projections (bf16 weights by TMA, 4-bit
    # codes expanded in shared memory)
    ("tc_decode_bf16_b4", synthetic.BF16, 4, 1, 2048),
    ("tc_decode_q4_b32", synthetic.AFFINE4_G64, 32, 1, 2048),
]


@pytest.fixture(scope="module")
def glue():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import torch_glue
    return torch_glue


def _case(name, fmt, batch, tps, hidden):
    wl = synthetic.custom(name=name, seed=sum(map(ord, name)), weight_format=fmt, batch=batch, hidden=hidden,
                          intermediate=2 * hidden, n_q_heads=4, n_kv_heads=2, head_dim=64, vocab=3000,
                          prefill=(0, 40) if batch > 1 else 40, steps=tps, n_layers=1)
    return wl, synthetic.generate(wl, device="cuda")


def _step(glue, wl, model, tps, kv):
    """One step (tokens_per_seq = tps) on a copy of the cache; returns logits, argmax."""
    rows = wl.batch * tps
    g = torch.Generator(device="cpu")
    g.manual_seed(7)
    toks = torch.randint(0, wl.vocab, (rows,), generator=g, dtype=torch.int32).cuda()
    if tps == 1:
        toks = model["tokens"]
    proj = 2 if wl.name.startswith("tc_decode") else 0
    dec = glue.Decoder(wl, model, tokens_per_seq=tps, proj_kernels=proj)
    try:
        logits = torch.empty((rows, wl.vocab), dtype=torch.float32, device="cuda")
        am = torch.empty((rows,), dtype=torch.int32, device="cuda")
        dec.step(toks, model["positions"], kv.clone(), logits, am)
        torch.cuda.synchronize()
        assert dec.device_status()[1] == 0
    finally:
        dec.close()
    return logits.cpu().numpy(), am.cpu().numpy()


def _consistent(logits, am, where):
    for r in range(logits.shape[0]):
        assert int(am[r]) == int(np.argmax(logits[r])), f"{where} row {r}: argmax {int(am[r])}, logits say " \
                                                       f"{int(np.argmax(logits[r]))}"


@pytest.mark.parametrize("name,fmt,batch,tps,hidden", CASES, ids=[c[0] for c in CASES])
def test_all_zero_lm_head_ties_everywhere(glue, name, fmt, batch, tps, hidden):
    wl, model = _case(name, fmt, batch, tps, hidden)
    if fmt == synthetic.BF16:
        model["lm_head"].zero_()
    else:
        model["lm_head"]["scales"].zero_()
        model["lm_head"]["biases"].zero_()
    logits, am = _step(glue, wl, model, tps, model["kv"])
    assert np.all(logits == 0.0)
    assert np.all(am == 0), f"argmax {am[am != 0][:5]} instead of 0"


@pytest.mark.parametrize("name,fmt,batch,tps,hidden", CASES, ids=[c[0] for c in CASES])
def test_copied_winner_row_ties_across_tiles(glue, name, fmt, batch, tps, hidden):
    wl, model = _case(name, fmt, batch, tps, hidden)
    kv0 = model["kv"].clone()
    logits, am = _step(glue, wl, model, tps, kv0)
    _consistent(logits, am, f"{name} first run")
    r0 = wl.batch * tps - 1  # the last row: for a prefill chunk, the row that yields the next token
    a = int(am[r0])
    if name == "tc_decode_bf16_b4":
        # the stream-K schedule splits tiles at K offsets that differ from tile to tile, so a
        # copy in another tile may round differently: the copies go to other warps and lanes of
        # the winner's own 128-row tile (the same MMAs and segments; ties across CTAs are the
        # all-zero test's)
        copies = [a ^ m for m in (1, 32, 64, 96) if (a ^ m) < wl.vocab]
    else:
        copies = [a + 256 * j for j in range(-7, 8) if j != 0 and 0 <= a + 256 * j < wl.vocab]
    assert len(copies) >= 3
    want = min(copies + [a])  # the lowest index among the tied rows
    lm = model["lm_head"]
    for c in copies:
        if fmt == synthetic.BF16:
            lm[c].copy_(lm[a])
        else:
            for k in ("w", "scales", "biases"):
                lm[k][c].copy_(lm[k][a])
    logits2, am2 = _step(glue, wl, model, tps, kv0)
    # the copies took the same arithmetic: bit-identical logits, an exact tie at the top
    for c in copies:
        assert logits2[r0, c] == logits2[r0, a], f"{name}: copy {c} gives {logits2[r0, c]!r}, row {a} " \
                                                 f"{logits2[r0, a]!r}"
    assert logits2[r0, a] == logits[r0, a]
    assert int(am2[r0]) == want, f"{name}: argmax {int(am2[r0])} among tied rows {sorted([a] + copies)}"
    _consistent(logits2, am2, f"{name} with copies")

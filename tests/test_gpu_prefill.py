"""Chunked prefill: one step with tokens_per_seq = T well beyond the batched path's
per-CTA token count (the projections run in token blocks) must be, row by row, the
one-token steps of the oracle with those tokens fed in (its verify_step: T teacher-
forced decode steps), with every appended K/V slot within two bf16 steps of the
oracle's (or, for the 8-bit cache, within one level) and every other slot untouched."""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import check_logits, kv_appended_close, np_model

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def glue():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import torch_glue
    return torch_glue


CASES = [
    # name, T, workload kwargs: bf16 blocks are 16 tokens, 4-bit blocks 32
    ("pf_b1_t40_bf16", 40, dict(batch=1, head_dim=128, n_q_heads=4, n_kv_heads=2, hidden=256, intermediate=512,
                                prefill=0, n_layers=2, vocab=700)),
    ("pf_b2_t37_bf16_ragged", 37, dict(batch=2, head_dim=64, n_q_heads=4, n_kv_heads=1, hidden=192,
                                       intermediate=384, prefill=(5, 90), n_layers=2, vocab=500)),
    ("pf_b3_t70_q4", 70, dict(batch=3, weight_format=synthetic.AFFINE4_G64, head_dim=128, n_q_heads=8, n_kv_heads=2,
                              hidden=256, intermediate=512, prefill=(0, 40), n_layers=2, vocab=600)),
    ("pf_b1_t129_q4_kv8", 129, dict(batch=1, weight_format=synthetic.AFFINE4_G64, head_dim=64, n_q_heads=4,
                                    n_kv_heads=2, hidden=320, intermediate=640, prefill=3, n_layers=2, vocab=400,
                                    kv_format=synthetic.AFFINE8_G64)),
    # the causal prefill attention (16+ tokens, bf16 cache): one query head per KV head with a
    # ragged last query tile; a chunk after a long cached prompt (many unmasked K/V tiles); the
    # smallest chunk that takes it
    ("pf_b2_t50_g1_bf16", 50, dict(batch=2, head_dim=64, n_q_heads=2, n_kv_heads=2, hidden=128, intermediate=256,
                                   prefill=(60, 130), n_layers=1, vocab=300)),
    ("pf_b1_t64_long_ctx", 64, dict(batch=1, head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=256,
                                    intermediate=512, prefill=3000, n_layers=1, vocab=300)),
    ("pf_b3_t16_g4", 16, dict(batch=3, head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=256, intermediate=512,
                              prefill=(0, 70), n_layers=1, vocab=300)),
    # 128 rows or more with bf16 weights and hidden >= 2048: the tcgen05 projections (ragged token
    # and weight tiles, a vocabulary that is not a multiple of 4)
    ("pf_b1_t200_bf16_tc5", 200, dict(batch=1, head_dim=128, n_q_heads=4, n_kv_heads=2, hidden=2048,
                                      intermediate=2112, prefill=0, n_layers=2, vocab=777)),
    ("pf_b2_t130_bf16_tc5_ragged", 130, dict(batch=2, head_dim=64, n_q_heads=8, n_kv_heads=2, hidden=2240,
                                             intermediate=1024, prefill=(5, 90), n_layers=2, vocab=500)),
    # gate/up (19456 rows) and lm_head (vocabulary 20000) fill the GPU with 256-row weight tiles
    ("pf_b2_t128_bf16_tc5_wide", 128, dict(batch=2, head_dim=64, n_q_heads=4, n_kv_heads=2, hidden=2048,
                                           intermediate=9728, prefill=(0, 30), n_layers=1, vocab=20000)),
    ("pf_b1_t160_bf16_tc5_kv8", 160, dict(batch=1, head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=2048,
                                          intermediate=1024, prefill=40, n_layers=2, vocab=1000,
                                          kv_format=synthetic.AFFINE8_G64)),
]


@pytest.mark.parametrize("name,T,kw", CASES, ids=[c[0] for c in CASES])
def test_prefill_matches_oracle(glue, name, T, kw):
    wl = synthetic.custom(name=name, seed=sum(map(ord, name)), steps=T, **kw)
    model = synthetic.generate(wl, device="cuda")
    host = synthetic.to_host(model)
    kv8 = wl.kv_format == synthetic.AFFINE8_G64
    if kv8:
        from test_gpu_kv8 import appended_rows_valid, host_cache, split_flat
        kv_init = host_cache(host["kv"])
        kv_dev = synthetic.kv_buffer(model["kv"])
    else:
        kv_init = np_model({"kv": host["kv"]})["kv"]
        kv_dev = model["kv"]
    B, V = wl.batch, wl.vocab
    g = torch.Generator(device="cpu")
    g.manual_seed(T)
    toks = torch.randint(0, V, (B, T), generator=g, dtype=torch.int32)
    dec = glue.Decoder(wl, model, tokens_per_seq=T)
    try:
        logits = torch.empty((B * T, V), dtype=torch.float32, device="cuda")
        argmax = torch.empty((B * T,), dtype=torch.int32, device="cuda")
        dec.step(toks.reshape(-1).cuda(), model["positions"], kv_dev, logits, argmax)
        torch.cuda.synchronize()
        assert dec.device_status()[1] == 0
        lg = logits.cpu().numpy().reshape(B, T, V)
        am = argmax.cpu().numpy().reshape(B, T)
        kv_out = kv_dev.cpu()
    finally:
        dec.close()
    m = oracle.OracleModel.from_synthetic(wl, host)
    kv_ref = kv_init.copy()
    ref_lg, ref_am = oracle.verify_step(m, kv_ref, toks.numpy(), host["positions"].numpy())
    for t in range(T):
        check_logits(lg[:, t], ref_lg[:, t], am[:, t], ref_am[:, t], f"{name} token {t}")
    if kv8:
        codes, params = split_flat(kv_out.numpy(), wl.n_layers, B, wl.n_kv_heads, wl.max_ctx, wl.head_dim)
        appended_rows_valid(oracle.Affine8Cache(codes, params), kv_ref, kv_init)
    else:
        kv_appended_close(np_model({"kv": kv_out})["kv"], kv_ref, kv_init)


def test_prefill_then_decode_continues_the_sequence(glue):
    """A prefill chunk followed by one-token steps gives the same greedy tokens and logits
    (within the tolerance) as one-token steps over the whole prompt."""
    wl = synthetic.custom(name="pf_then_decode", seed=91, batch=2, head_dim=64, n_q_heads=4, n_kv_heads=2,
                          hidden=192, intermediate=384, prefill=(0, 20), n_layers=2, vocab=300, steps=40)
    T = 33
    g = torch.Generator(device="cpu")
    g.manual_seed(5)
    toks = torch.randint(0, wl.vocab, (wl.batch, T), generator=g, dtype=torch.int32)
    model = synthetic.generate(wl, device="cuda")
    B, V = wl.batch, wl.vocab
    # (a) one prefill step of T tokens
    kv_a = model["kv"].clone()
    pf = glue.Decoder(wl, model, tokens_per_seq=T)
    la = torch.empty((B * T, V), device="cuda")
    aa = torch.empty((B * T,), dtype=torch.int32, device="cuda")
    pf.step(toks.reshape(-1).cuda(), model["positions"], kv_a, la, aa)
    pf.close()
    # (b) T one-token steps with the same tokens
    kv_b = model["kv"].clone()
    one = glue.Decoder(wl, model)
    lb = torch.empty((B, V), device="cuda")
    ab = torch.empty((B,), dtype=torch.int32, device="cuda")
    pos = model["positions"].clone()
    rows = []
    for t in range(T):
        one.step(toks[:, t].contiguous().cuda(), pos, kv_b, lb, ab)
        pos += 1
        rows.append(lb.cpu().numpy().copy())
    one.close()
    torch.cuda.synchronize()
    la_h = la.cpu().numpy().reshape(B, T, V)
    for t in range(T):
        d = np.abs(la_h[:, t] - rows[t])
        assert float(d.max()) < 5e-3, f"token {t}: prefill and one-token logits differ by {float(d.max()):.3e}"


def test_tc5_weights_dequant_bit_exact(glue):
    """The row-major packing of the tcgen05 path (gate/up interleaved in blocks of 16) through
    dec_debug_dequant: every linear equals its bf16 source exactly."""
    from oracle import numerics
    wl = synthetic.custom(name="dq5", head_dim=64, n_q_heads=4, n_kv_heads=2, hidden=2048, intermediate=320,
                          vocab=200, n_layers=2, batch=1, steps=130)
    model = synthetic.generate(wl, device="cuda", with_kv=False)
    host = np_model(synthetic.to_host(model))
    dec = glue.Decoder(wl, model, tokens_per_seq=130)
    names = ["q", "k", "v", "o", "gate", "up", "down", "lm_head"]
    try:
        for layer in range(wl.n_layers):
            for which, name in enumerate(names):
                if which == 7 and layer > 0:
                    continue
                src = host["lm_head"] if which == 7 else host["layers"][layer][name]
                ref = numerics.bf16_bits_to_f64(src).astype(np.float32)
                out = torch.empty(ref.shape, dtype=torch.float32, device="cuda")
                dec.debug_dequant(layer, which, out)
                assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32)), f"layer {layer} {name}"
    finally:
        dec.close()

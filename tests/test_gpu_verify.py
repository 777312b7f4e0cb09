"""Multi-token verify step (tokens_per_seq T > 1) against the oracle's verify_step:
row (b, t) must be the one-token step of sequence b at position P_b + t after the
rows (b, 0..t-1), under the same logits tolerance as a decode step, with the step's
T K/V slots per sequence within two bf16 steps and every other slot untouched."""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import check_logits, kv_appended_close, np_model

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def glue():
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import torch_glue
    return torch_glue


CASES = [
    # name, T, workload kwargs (rows = batch * T within the batched limits)
    ("v_b1_t4_bf16", 4, dict(batch=1, head_dim=128, n_q_heads=4, n_kv_heads=2, hidden=256, intermediate=512,
                             prefill=70, n_layers=2)),
    ("v_b2_t8_bf16", 8, dict(batch=2, head_dim=64, n_q_heads=4, n_kv_heads=1, hidden=192, intermediate=384,
                             prefill=(3, 130), n_layers=2)),
    ("v_b3_t5_q4", 5, dict(batch=3, weight_format="affine4_g64", head_dim=64, n_q_heads=2, n_kv_heads=1,
                           hidden=256, intermediate=512, prefill=(0, 200), n_layers=2)),
    ("v_b1_t2_q4", 2, dict(batch=1, weight_format="affine4_g64", head_dim=128, n_q_heads=8, n_kv_heads=2,
                           hidden=512, intermediate=1024, prefill=513, n_layers=1)),
]


def _verify(glue, wl, T, graph):
    model = synthetic.generate(wl, device="cuda")
    host = synthetic.to_host(model)
    kv_init = np_model({"kv": host["kv"]})["kv"]
    B, V = wl.batch, wl.vocab
    g = torch.Generator(device="cpu")
    g.manual_seed(len(wl.name) * 31 + T)
    toks = torch.randint(0, V, (B, T), generator=g, dtype=torch.int32)
    dec = glue.Decoder(wl, model, tokens_per_seq=T)
    dec.set_graph_mode(graph)
    try:
        logits = torch.empty((B * T, V), dtype=torch.float32, device="cuda")
        argmax = torch.empty((B * T,), dtype=torch.int32, device="cuda")
        kv = model["kv"]
        dec.step(toks.reshape(-1).cuda(), model["positions"], kv, logits, argmax)
        torch.cuda.synchronize()
        assert dec.device_status()[1] == 0
        lg = logits.cpu().numpy().reshape(B, T, V)
        am = argmax.cpu().numpy().reshape(B, T)
        kv_gpu = np_model({"kv": kv.cpu()})["kv"]
    finally:
        dec.close()
    m = oracle.OracleModel.from_synthetic(wl, host)
    kv_ref = kv_init.copy()
    ref_lg, ref_am = oracle.verify_step(m, kv_ref, toks.numpy(), host["positions"].numpy())
    return lg, am, ref_lg, ref_am, kv_gpu, kv_ref, kv_init


@pytest.mark.parametrize("name,T,kw", CASES)
def test_verify_matches_oracle(glue, name, T, kw):
    wl = synthetic.custom(name=name, seed=sum(map(ord, name)), steps=T, **kw)
    lg, am, ref_lg, ref_am, kv_gpu, kv_ref, kv_init = _verify(glue, wl, T, graph=True)
    for t in range(T):
        check_logits(lg[:, t], ref_lg[:, t], am[:, t], ref_am[:, t], f"{name} token {t}")
    kv_appended_close(kv_gpu, kv_ref, kv_init)


def test_verify_graph_equals_eager(glue):
    name, T, kw = CASES[0]
    wl = synthetic.custom(name=name, seed=7, steps=T, **kw)
    a = _verify(glue, wl, T, graph=True)
    b = _verify(glue, wl, T, graph=False)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[4], b[4])


def test_verify_rows_agree_with_one_token_steps(glue):
    """The verify rows against the GPU's own one-token steps fed the same tokens
    (different projection kernels: same tolerance as against the oracle)."""
    name, T, kw = "v_vs_decode", 4, dict(batch=1, head_dim=64, n_q_heads=2, n_kv_heads=1, hidden=128,
                                          intermediate=256, prefill=40, n_layers=2)
    wl = synthetic.custom(name=name, seed=11, steps=T, **kw)
    lg, am, _, _, kv_v, _, _ = _verify(glue, wl, T, graph=True)
    model = synthetic.generate(wl, device="cuda")
    g = torch.Generator(device="cpu")
    g.manual_seed(len(wl.name) * 31 + T)
    toks = torch.randint(0, wl.vocab, (1, T), generator=g, dtype=torch.int32)
    dec = glue.Decoder(wl, model)
    try:
        pos = model["positions"].clone()
        out = torch.empty((1, wl.vocab), dtype=torch.float32, device="cuda")
        a1 = torch.empty((1,), dtype=torch.int32, device="cuda")
        for t in range(T):
            dec.step(toks[:, t].contiguous().cuda(), pos, model["kv"], out, a1)
            torch.cuda.synchronize()
            check_logits(lg[:, t], out.cpu().numpy().astype(np.float64), am[:, t], a1.cpu().numpy(),
                         f"verify vs decode token {t}")
            pos += 1
    finally:
        dec.close()


def test_verify_rejects_too_many_rows(glue):
    from token_decode_step_gb300 import dec as D
    wl = synthetic.custom(name="v_big", batch=17, steps=8)
    model = synthetic.generate(wl, device="cuda", with_kv=False)  # 17 x 4000 rows > 65535
    with pytest.raises(D.DecError) as ei:
        glue.Decoder(wl, model, tokens_per_seq=4000)
    assert "rows" in str(ei.value)
    with pytest.raises(D.DecError) as ei:
        glue.Decoder(wl, model, tokens_per_seq=4097)
    assert "tokens_per_seq" in str(ei.value)

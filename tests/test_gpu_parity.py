"""GPU parity: the CUDA decode step (through the C ABI) against the CPU oracle on
the same seeded inputs.  Needs a GB300 (sm_103a)."""

import numpy as np
import pytest
import torch

import synthetic
from parity import check_logits, gpu_greedy, kv_appended_close, np_model, oracle_replay

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def glue():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import torch_glue
    return torch_glue


def _run(glue, wl, steps, check_steps=None, graph=True):
    model = synthetic.generate(wl, device="cuda")
    host = synthetic.to_host(model)
    kv_init = np_model({"kv": host["kv"]})["kv"]
    dec = glue.Decoder(wl, model)
    dec.set_graph_mode(graph)
    try:
        gpu_steps, kv = gpu_greedy(dec, model, steps)
        st, bits = dec.device_status()
        assert bits == 0, f"device status bits {bits}"
    finally:
        dec.close()
    res, kv_ref = oracle_replay(wl, host, kv_init, gpu_steps, check_steps)
    worst = {"max_abs": 0.0, "rel_l2": 0.0, "exempt": 0}
    for s, lg, am in res:
        w = check_logits(gpu_steps[s][2], lg, gpu_steps[s][3], am, f"{wl.name} step {s}")
        worst = {k: max(worst[k], w[k]) if k != "exempt" else worst[k] + w[k] for k in worst}
    if check_steps is None:
        kv_gpu = np_model({"kv": kv.cpu()})["kv"]
        kv_appended_close(kv_gpu, kv_ref, kv_init)
    return worst


def test_tiny_all_steps(glue):
    w = _run(glue, synthetic.WORKLOADS["tiny"], 16)
    print("tiny worst", w)


CUSTOM = [
    # name, overrides
    ("d64_g1_emptycache_ragged_vocab", dict(head_dim=64, n_q_heads=2, n_kv_heads=2, hidden=128, intermediate=256,
                                             vocab=1003, prefill=0, steps=3)),
    ("d128_g4_multi_split", dict(head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=256, intermediate=512, vocab=777,
                                 prefill=700, steps=3)),
    ("d128_g2_long_ctx", dict(head_dim=128, n_q_heads=4, n_kv_heads=2, hidden=192, intermediate=384, vocab=640,
                              prefill=3000, steps=2, n_layers=2)),
    ("q4_d128_g2", dict(weight_format=synthetic.AFFINE4_G64, head_dim=128, n_q_heads=4, n_kv_heads=2, hidden=256,
                        intermediate=512, vocab=500, prefill=130, steps=3, n_layers=2)),
    ("q4_d64_g4", dict(weight_format=synthetic.AFFINE4_G64, head_dim=64, n_q_heads=8, n_kv_heads=2, hidden=384,
                       intermediate=1024, vocab=2049, prefill=63, steps=3, n_layers=2)),
    ("bf16_tile_edge", dict(head_dim=128, n_q_heads=2, n_kv_heads=1, hidden=128, intermediate=192, vocab=64,
                            prefill=127, steps=3)),
]


@pytest.mark.parametrize("name,kw", CUSTOM, ids=[c[0] for c in CUSTOM])
def test_custom_shapes(glue, name, kw):
    wl = synthetic.custom(name=name, seed=hash(name) % 1000, **kw)
    w = _run(glue, wl, wl.steps)
    print(name, w)


def test_graph_equals_eager_bitwise(glue):
    wl = synthetic.WORKLOADS["tiny"]
    outs = []
    for graph in (True, False):
        model = synthetic.generate(wl, device="cuda")
        dec = glue.Decoder(wl, model)
        dec.set_graph_mode(graph)
        steps, _ = gpu_greedy(dec, model, 4)
        dec.close()
        outs.append(steps)
    for a, b in zip(*outs):
        assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])


def test_repeated_step_is_deterministic(glue):
    wl = synthetic.custom(name="det", head_dim=128, n_q_heads=4, n_kv_heads=1, hidden=256, intermediate=512,
                          vocab=999, prefill=900, steps=1)
    model = synthetic.generate(wl, device="cuda")
    dec = glue.Decoder(wl, model)
    logits = torch.empty((1, wl.vocab), device="cuda")
    am = torch.empty((1,), dtype=torch.int32, device="cuda")
    kv0 = model["kv"].clone()
    res = []
    for _ in range(3):
        model["kv"].copy_(kv0)
        dec.step(model["tokens"], model["positions"], model["kv"], logits, am)
        torch.cuda.synchronize()
        res.append(logits.cpu().clone())
    dec.close()
    assert torch.equal(res[0], res[1]) and torch.equal(res[0], res[2])


@pytest.mark.parametrize("fmt", [synthetic.BF16, synthetic.AFFINE4_G64])
def test_debug_dequant_bit_exact(glue, fmt):
    from oracle import affine4, numerics
    wl = synthetic.custom(name="dq", weight_format=fmt, head_dim=64, n_q_heads=4, n_kv_heads=2, hidden=192,
                          intermediate=320, vocab=200, n_layers=2)
    model = synthetic.generate(wl, device="cuda", with_kv=False)
    host = np_model(synthetic.to_host(model))
    dec = glue.Decoder(wl, model)
    names = ["q", "k", "v", "o", "gate", "up", "down", "lm_head"]
    try:
        for layer in range(wl.n_layers):
            for which, name in enumerate(names):
                if which == 7 and layer > 0:
                    continue
                src = host["lm_head"] if which == 7 else host["layers"][layer][name]
                if fmt == synthetic.BF16:
                    ref = numerics.bf16_bits_to_f64(src).astype(np.float32)
                else:
                    ref = affine4.dequant_affine4_g64_f32(src["w"].view(np.uint32), src["scales"], src["biases"])
                out = torch.empty(ref.shape, dtype=torch.float32, device="cuda")
                dec.debug_dequant(layer, which, out)
                got = out.cpu().numpy()
                assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"layer {layer} {name}"
    finally:
        dec.close()


def test_out_of_range_inputs_are_flagged(glue):
    wl = synthetic.custom(name="bad", vocab=300, prefill=10, steps=1)
    model = synthetic.generate(wl, device="cuda")
    dec = glue.Decoder(wl, model)
    logits = torch.empty((1, wl.vocab), device="cuda")
    am = torch.empty((1,), dtype=torch.int32, device="cuda")
    try:
        tok = torch.tensor([wl.vocab + 5], dtype=torch.int32, device="cuda")
        dec.step(tok, model["positions"], model["kv"], logits, am)
        torch.cuda.synchronize()
        st, bits = dec.device_status()
        assert bits == 1 and st == 6
        pos = torch.tensor([wl.max_ctx + 3], dtype=torch.int32, device="cuda")
        dec.step(model["tokens"], pos, model["kv"], logits, am)
        torch.cuda.synchronize()
        st, bits = dec.device_status()
        assert bits == 2 and st == 6
        assert torch.isfinite(logits).all()
        st, bits = dec.device_status()
        assert bits == 0 and st == 0
    finally:
        dec.close()


def test_qwen3_0_6b_first_steps(glue):
    wl = synthetic.WORKLOADS["qwen3-0.6b"]
    w = _run(glue, wl, 6)
    print("qwen3-0.6b worst", w)

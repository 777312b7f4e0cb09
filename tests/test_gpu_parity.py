"""GPU parity: the CUDA decode step (through the C ABI) against the CPU oracle on
the same seeded inputs.  Needs a GB300 (sm_103a)."""

import numpy as np
import pytest
import torch

import synthetic
import oracle
from parity import check_logits, gpu_greedy, kv_appended_close, np_model, oracle_replay, replay_plan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def glue():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import torch_glue
    return torch_glue


def _run(glue, wl, steps, graph=True, full_kv_check=True, cache_weights=True, plan=None, proj=0):
    """Greedy loop of `steps` steps on the GPU, then the oracle replays the GPU's tokens.

    plan: [(sequences or None for all, number of leading steps)] to replay (default: every
    sequence over every step).  Every replayed (step, sequence) must meet the tolerances;
    there is no exemption beyond the top-2 near tie of the argmax."""
    model = synthetic.generate(wl, device="cuda")
    host = synthetic.to_host(model)
    kv_init = np_model({"kv": host["kv"]})["kv"]
    dec = glue.Decoder(wl, model, proj_kernels=proj)
    dec.set_graph_mode(graph)
    try:
        gpu_steps, kv = gpu_greedy(dec, model, steps)
        st, bits = dec.device_status()
        assert bits == 0, f"device status bits {bits}"
    finally:
        dec.close()
    m = oracle.OracleModel.from_synthetic(wl, host, cache_weights=cache_weights)
    worst = {"max_abs": 0.0, "rel_l2": 0.0, "exempt": 0, "replayed": []}
    for seqs, n in plan or [(None, steps)]:
        res, kv_ref = oracle_replay(wl, host, kv_init, gpu_steps[:n], seqs=seqs, model=m)
        sel = slice(None) if seqs is None else np.asarray(seqs)
        for s, lg, am in res:
            w = check_logits(gpu_steps[s][2][sel], lg, gpu_steps[s][3][sel], am,
                             f"{wl.name} step {s} seqs {'all' if seqs is None else list(seqs)}")
            worst["max_abs"] = max(worst["max_abs"], w["max_abs"])
            worst["rel_l2"] = max(worst["rel_l2"], w["rel_l2"])
            worst["exempt"] += w["exempt"]
        worst["replayed"].append(("all" if seqs is None else list(seqs), n))
        if full_kv_check and seqs is None and n == steps:
            kv_gpu = np_model({"kv": kv.cpu()})["kv"]
            kv_appended_close(kv_gpu, kv_ref, kv_init)
        else:  # the slots the replayed steps appended (the full cache is tens of GB)
            idx = range(wl.batch) if seqs is None else seqs
            for _, pin, _, _ in gpu_steps[:n]:
                for j, b in enumerate(idx):
                    P = int(pin[b])
                    g = np_model({"kv": kv[:, :, b, :, P].cpu()})["kv"]
                    appended_vectors_close(g, kv_ref[:, :, j, :, P], f"{wl.name} seq {b} slot {P}")
    return worst


def appended_vectors_close(gpu_bits, ref_bits, where):
    """Appended K/V vectors (last axis head_dim): max |gpu - ref| <= 2 * 2^-8 * max |ref|."""
    from oracle import numerics
    g = numerics.bf16_bits_to_f64(gpu_bits)
    r = numerics.bf16_bits_to_f64(ref_bits)
    err = np.max(np.abs(g - r), axis=-1)
    scale = np.max(np.abs(r), axis=-1)
    assert np.all(err <= 2 * 2.0 ** -8 * scale), f"{where}: appended K/V off by {float(np.max(err / scale)):.3g}"


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
    # 4-bit at batch 1, hidden 2048 (the tcgen05 paths start at 2 rows)
    ("q4_b1_h2048", dict(weight_format=synthetic.AFFINE4_G64, head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=2048,
                       intermediate=2880, vocab=1500, prefill=300, steps=3, n_layers=2)),
]


CUSTOM_BATCHED = [
    ("b3_bf16_ragged", dict(batch=3, prefill=(0, 300), head_dim=128, n_q_heads=4, n_kv_heads=2, hidden=256,
                            intermediate=512, vocab=1000, steps=3, n_layers=2)),
    ("b12_bf16", dict(batch=12, prefill=(10, 200), head_dim=64, n_q_heads=8, n_kv_heads=2, hidden=192,
                      intermediate=384, vocab=517, steps=2, n_layers=2)),
    ("b5_q4", dict(batch=5, weight_format=synthetic.AFFINE4_G64, prefill=(1, 700), head_dim=128, n_q_heads=8,
                   n_kv_heads=2, hidden=256, intermediate=640, vocab=999, steps=3, n_layers=2)),
    ("b20_q4", dict(batch=20, weight_format=synthetic.AFFINE4_G64, prefill=(0, 1500), head_dim=64, n_q_heads=4,
                    n_kv_heads=1, hidden=320, intermediate=768, vocab=2000, steps=2, n_layers=2)),
    # 32 rows of 4-bit weights at hidden >= 2048, mma.sync selected explicitly (proj 1)
    ("b32_q4_long_k", dict(proj=1, batch=32, weight_format=synthetic.AFFINE4_G64, prefill=(100, 400), head_dim=128,
                           n_q_heads=4, n_kv_heads=1, hidden=2560, intermediate=4096, vocab=333, steps=2,
                           n_layers=1)),
    ("b8_bf16_long_k", dict(batch=8, prefill=(50, 300), head_dim=128, n_q_heads=4, n_kv_heads=2, hidden=4096,
                            intermediate=6144, vocab=700, steps=2, n_layers=1)),
    # hidden >= 2048, at most 32 rows, the tcgen05 decode projections selected (proj 2): 4-bit
    # codes expanded in shared memory, bf16 weights streamed by TMA
    ("b3_q4_tc5", dict(proj=2, batch=3, weight_format=synthetic.AFFINE4_G64, prefill=(0, 200), head_dim=128, n_q_heads=8,
                       n_kv_heads=2, hidden=2048, intermediate=2880, vocab=1234, steps=2, n_layers=2)),
    ("b20_q4_tc5", dict(proj=2, batch=20, weight_format=synthetic.AFFINE4_G64, prefill=(5, 600), head_dim=64, n_q_heads=16,
                        n_kv_heads=4, hidden=2048, intermediate=5632, vocab=3001, steps=2, n_layers=1)),
    ("b8_bf16_tc5", dict(proj=2, batch=8, prefill=(50, 300), head_dim=128, n_q_heads=4, n_kv_heads=2, hidden=2048,
                         intermediate=3072, vocab=1100, steps=2, n_layers=2)),
    ("b32_q4_tc5_long_k", dict(proj=2, batch=32, weight_format=synthetic.AFFINE4_G64, prefill=(100, 400),
                               head_dim=128, n_q_heads=4, n_kv_heads=1, hidden=2560, intermediate=4096, vocab=333,
                               steps=2, n_layers=1)),
]


@pytest.mark.parametrize("name,kw", CUSTOM_BATCHED, ids=[c[0] for c in CUSTOM_BATCHED])
def test_custom_batched(glue, name, kw):
    kw = dict(kw)
    proj = kw.pop("proj", 0)
    wl = synthetic.custom(name=name, seed=sum(map(ord, name)), **kw)
    w = _run(glue, wl, wl.steps, proj=proj)
    print(name, w)


@pytest.mark.parametrize("name,kw", CUSTOM, ids=[c[0] for c in CUSTOM])
def test_custom_shapes(glue, name, kw):
    wl = synthetic.custom(name=name, seed=sum(map(ord, name)), **kw)  # stable across processes
    w = _run(glue, wl, wl.steps)
    print(name, w)


@pytest.mark.parametrize("batch", [1, 4])
def test_graph_equals_eager_bitwise(glue, batch):
    wl = synthetic.WORKLOADS["tiny"].replace(batch=batch)
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


@pytest.mark.parametrize("batch,graph", [(1, True), (4, True), (4, False)])
def test_host_step_equals_device_step_bitwise(glue, batch, graph):
    """dec_step_host (host token ids, positions and argmax, copies inside the call) gives
    the device-pointer step's logits, argmax and appended K/V bit for bit; its argmax
    output aliases its token input, the host greedy loop's natural form."""
    wl = synthetic.WORKLOADS["tiny"].replace(batch=batch)
    model = synthetic.generate(wl, device="cuda")
    dec = glue.Decoder(wl, model)
    dec.set_graph_mode(graph)
    kv0 = model["kv"].clone()
    try:
        ref, kv_ref = gpu_greedy(dec, model, 4)
        kv_ref = kv_ref.clone()
        model["kv"].copy_(kv0)
        tok = model["tokens"].cpu().numpy().astype(np.int32).copy()
        pos = model["positions"].cpu().numpy().astype(np.int32).copy()
        logits = torch.empty((batch, wl.vocab), device="cuda")
        for s, (tin, pin, lg, am) in enumerate(ref):
            assert np.array_equal(tok, tin) and np.array_equal(pos, pin), f"step {s} inputs"
            dec.step_host(tok, pos, model["kv"], logits, tok)
            assert np.array_equal(tok, am), f"step {s} argmax"
            assert np.array_equal(logits.cpu().numpy(), lg), f"step {s} logits"
            pos += 1
        torch.cuda.synchronize()
        assert torch.equal(model["kv"], kv_ref)
        assert dec.device_status()[1] == 0
    finally:
        dec.close()


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


@pytest.mark.parametrize("batch,hidden", [(1, 192), (6, 192), (4, 2048)])
@pytest.mark.parametrize("fmt", [synthetic.BF16, synthetic.AFFINE4_G64])
def test_debug_dequant_bit_exact(glue, fmt, batch, hidden):
    """Every packing (batch 1; batched mma.sync fragments; at hidden 2048 the 4-bit batched
    tcgen05 path's row-major packing) reads back the caller's weights bit for bit."""
    from oracle import affine4, numerics
    wl = synthetic.custom(name="dq", weight_format=fmt, head_dim=64, n_q_heads=4, n_kv_heads=2, hidden=hidden,
                          intermediate=320, vocab=200, n_layers=2, batch=batch)
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


def test_forced_timeout_is_reported_and_the_handle_stays_usable(glue):
    """A bounded device wait that can only run out (an mbarrier nothing arrives on) sets the
    time-out bit; dec_get_device_status reports DEC_ERR_TIMEOUT once and clears it, and the next
    step runs normally.  No fault or trap is involved."""
    from token_decode_step_gb300 import dec as D
    wl = synthetic.WORKLOADS["tiny"]
    model = synthetic.generate(wl, device="cuda")
    dec = glue.Decoder(wl, model)
    logits = torch.empty((1, wl.vocab), device="cuda")
    am = torch.empty((1,), dtype=torch.int32, device="cuda")
    try:
        D.dec_debug_force_timeout(dec.handle, 256, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        st, bits = dec.device_status()
        assert st == D.DEC_ERR_TIMEOUT and bits & 4
        assert dec.device_status() == (0, 0)
        dec.step(model["tokens"], model["positions"], model["kv"], logits, am)
        torch.cuda.synchronize()
        assert dec.device_status() == (0, 0) and torch.isfinite(logits).all()
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


@pytest.mark.parametrize("name", ["qwen3-0.6b", "qwen3-4b-q4", "qwen3-8b-b1", "qwen3-8b-b8", "qwen3-8b-q4-b32"])
def test_full_size_all_steps(glue, name):
    """Full-size configs in the launch configuration the bench times (CUDA graph, same batch
    and cache), every greedy step of the config against the oracle: batch 1 over all steps;
    batches 8 and 32 over all steps for three fixed sequences and over the first two steps
    for every sequence (the sequences of a batch are independent)."""
    wl = synthetic.WORKLOADS[name]
    w = _run(glue, wl, wl.steps, full_kv_check=False, plan=replay_plan(wl))
    print(name, "worst", w)

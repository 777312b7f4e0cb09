"""GPU parity of the affine 8-bit KV cache (dec_config.kv_fmt = DEC_KV_AFFINE8_G64):
the quantizer bit-exact against the oracle's, the attention kernel and whole steps
against the oracle over a quantized cache.

Where the two sides quantize values they computed differently (the appended K comes from
float32 norm and RoPE on the GPU, float64 in the oracle; at step level also V), a value
that lies on a rounding boundary may take the neighbouring code, or the group's bf16 scale
or bias the neighbouring value: both are correct quantizations.  Appended rows are
therefore checked for validity (within one level of the oracle's row) plus a floor on how
many codes agree exactly; the attention output of a sequence whose appended K row took
such a neighbouring code is held to the loose step tolerance instead of the kernel one."""

import pathlib

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import numerics
from parity import ATTN_ATOL, ATTN_RTOL, check_logits, gpu_greedy, np_model, oracle_replay, replay_plan

pytestmark = pytest.mark.gpu

GOLDEN = pathlib.Path(__file__).parent / "golden"


@pytest.fixture(scope="module")
def glue():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import torch_glue
    return torch_glue


# ------------------------------------------------------------------ the quantizer

def _golden_rows():
    rows = []
    for line in (GOLDEN / "affine8_kv_worked_examples.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        _, fill, vals, _, _, _ = [f.strip() for f in line.split("|")]
        x = np.full(64, float(fill), dtype=np.float32)
        for kv in vals.split():
            i, v = kv.split("=")
            x[int(i)] = np.float32(float(v))
        rows.append(x)
    return np.stack(rows)


@pytest.mark.parametrize("d", [64, 128])
def test_kv_quantize_bit_exact(glue, d):
    rng = np.random.default_rng(d)
    n = 3000
    loc = rng.standard_normal((n, 1)) * 4
    spread = np.exp(rng.uniform(-8, 4, (n, 1)))
    x = (loc + spread * rng.standard_normal((n, d))).astype(np.float32)
    x[5, :] = 1.25                                   # constant row: scale 0, codes 0
    x[6, : d // 2] = -3.0                            # one constant group, one spread group
    x[7] = np.round(x[7] * 4) / 4                    # values on a coarse grid (exact ties)
    gold = _golden_rows()                            # the hand-worked groups
    x[8: 8 + len(gold) * 64 // d] = np.resize(gold, (len(gold) * 64 // d, d))
    src = torch.from_numpy(x).cuda()
    codes = torch.empty((n, d), dtype=torch.uint8, device="cuda")
    params = torch.empty((n, d // 64, 2), dtype=torch.bfloat16, device="cuda")
    glue.kv_quantize(src, codes, params)
    torch.cuda.synchronize()
    c_ref, s_ref, b_ref = oracle.quantize_affine8_g64(x)
    p = params.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert np.array_equal(p[..., 0], s_ref)
    assert np.array_equal(p[..., 1], b_ref)


# ------------------------------------------------------------------ cache helpers

def split_flat(flat: np.ndarray, L, B, nkv, max_ctx, d):
    """The library's flat kv8 buffer -> (codes uint8 [L][2][B][nkv][max_ctx][d],
    params uint16 [L][2][B][nkv][max_ctx][d/64][2])."""
    n = L * 2 * B * nkv * max_ctx * d
    off = (n + 255) // 256 * 256
    codes = flat[:n].reshape(L, 2, B, nkv, max_ctx, d)
    params = flat[off: off + n // 64 * 4].view(np.uint16).reshape(L, 2, B, nkv, max_ctx, d // 64, 2)
    return codes, params


def host_cache(kv: dict) -> oracle.Affine8Cache:
    return oracle.Affine8Cache(kv["codes"].cpu().numpy().copy(),
                               kv["params"].cpu().view(torch.int16).numpy().view(np.uint16).copy())


def appended_rows_valid(gpu: oracle.Affine8Cache, ref: oracle.Affine8Cache, init: oracle.Affine8Cache,
                        min_exact: float = 0.99) -> int:
    """Untouched slots bit-identical; every appended row (one head, one slot, K or V) within
    one quantization level of the oracle's (plus the bf16 step of the row's scale); at
    least `min_exact` of the appended codes equal.  Returns the number of rows whose codes
    or pairs differ."""
    ch = (np.any(gpu.codes != init.codes, axis=-1) | np.any(ref.codes != init.codes, axis=-1) |
          np.any(gpu.params != init.params, axis=(-1, -2)) | np.any(ref.params != init.params, axis=(-1, -2)))
    assert np.array_equal(gpu.codes[~ch], init.codes[~ch])
    assert np.array_equal(gpu.params[~ch], init.params[~ch])
    gc, gp = gpu.codes[ch], gpu.params[ch]
    rc, rp = ref.codes[ch], ref.params[ch]
    g = oracle.dequant_affine8_g64(gc, gp[..., 0], gp[..., 1])
    r = oracle.dequant_affine8_g64(rc, rp[..., 0], rp[..., 1])
    s = np.maximum(numerics.bf16_bits_to_f64(gp[..., 0]), numerics.bf16_bits_to_f64(rp[..., 0]))
    s = np.repeat(s, 64, axis=-1)
    scale = np.max(np.abs(r), axis=-1, keepdims=True)
    err = np.abs(g - r)
    assert np.all(err <= 1.01 * s + 2.0 ** -7 * scale), f"appended row off by {float(np.max(err / (s + 1e-30))):.3g} levels"
    exact = float(np.mean(gc == rc))
    assert exact >= min_exact, f"only {exact:.4f} of the appended codes equal the oracle's"
    return int(np.sum(np.any(gc != rc, axis=-1) | np.any(gp != rp, axis=(-1, -2))))


# ------------------------------------------------------------------ the attention kernel

ATT_CASES = [
    # B, nq, nkv, d, positions, max_ctx
    (1, 16, 8, 128, [1024], 1152),
    (3, 8, 2, 64, [0, 65, 700], 800),
    (2, 32, 8, 128, [4095, 513], 4160),
    (4, 4, 4, 128, [2000, 1, 64, 127], 2080),
    (2, 8, 4, 64, [8191, 3], 8224),
    (6, 16, 4, 128, [1500, 0, 63, 64, 777, 1200], 1536),
    (12, 4, 2, 64, [5, 300, 17, 1000, 64, 129, 2, 999, 640, 31, 1023, 256], 1024),
    (10, 16, 4, 128, [900, 1, 2047, 333, 64, 65, 1500, 0, 1000, 2000], 2048),
    # the batch-32 8B shapes: 256 clusters (several waves of two CTAs per SM), long contexts
    (32, 32, 8, 128, [int(x) for x in np.random.default_rng(32).integers(512, 8193, 32)], 8224),
]


def _kv8_case(seed, B, nkv, d, max_ctx, L=2):
    wl = synthetic.custom(name="att", seed=seed, n_layers=L, n_kv_heads=nkv, n_q_heads=nkv, head_dim=d,
                          batch=B, prefill=max_ctx - 1, steps=1, kv_format=synthetic.AFFINE8_G64)
    return synthetic.generate(wl)["kv"]


@pytest.mark.parametrize("B,nq,nkv,d,positions,max_ctx", ATT_CASES)
def test_kv8_attention_kernel_matches_oracle(glue, B, nq, nkv, d, positions, max_ctx):
    from token_decode_step_gb300 import dec
    g = torch.Generator(device="cpu")
    g.manual_seed(B * 1000 + d)
    qkv = torch.randn((B, (nq + 2 * nkv) * d), generator=g) * 0.7
    q_norm = (1 + 0.1 * torch.randn((d,), generator=g)).to(torch.bfloat16)
    k_norm = (1 + 0.1 * torch.randn((d,), generator=g)).to(torch.bfloat16)
    kv = _kv8_case(B * 7 + d, B, nkv, d, max_ctx)
    init = host_cache(kv)
    flat = synthetic.kv_buffer(kv).cuda()
    cfg = dec.DecConfig(n_layers=2, hidden=64, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, intermediate=64, vocab=1,
                        rms_eps=1e-6, rope_theta=1e6, linear_fmt=0, batch=B, max_ctx=max_ctx,
                        kv_fmt=dec.DEC_KV_AFFINE8_G64)
    ws_bytes = dec.dec_attention_workspace_bytes(cfg)
    ws = torch.empty((ws_bytes,), dtype=torch.uint8, device="cuda")
    out = torch.full((B, nq * d), float("nan"), device="cuda")
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    layer = 1
    d_qkv, d_qn, d_kn = qkv.cuda(), q_norm.cuda(), k_norm.cuda()
    dec.dec_attention(cfg, layer, d_qkv.data_ptr(), d_qn.data_ptr(), d_kn.data_ptr(), pos.data_ptr(),
                      flat.data_ptr(), out.data_ptr(), ws.data_ptr(), ws_bytes, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()

    # the oracle: the attention part of its step for one layer over the quantized cache
    ref_cache = init.copy()
    qn = numerics.bf16_bits_to_f64(q_norm.view(torch.int16).numpy().view(np.uint16))
    kn = numerics.bf16_bits_to_f64(k_norm.view(torch.int16).numpy().view(np.uint16))
    x = qkv.double().numpy()
    ref = np.empty((B, nq * d))
    for b in range(B):
        P = positions[b]
        q = oracle.rope_rotate_half(oracle.rmsnorm(x[b, : nq * d].reshape(nq, d), qn, 1e-6), P, 1e6)
        k = oracle.rope_rotate_half(oracle.rmsnorm(x[b, nq * d:(nq + nkv) * d].reshape(nkv, d), kn, 1e-6), P, 1e6)
        v = x[b, (nq + nkv) * d:].reshape(nkv, d)
        ref_cache.store(layer, 0, b, P, k)
        ref_cache.store(layer, 1, b, P, v)
        ref[b] = oracle.gqa_attention(q, ref_cache.read(layer, 0, b, P + 1), ref_cache.read(layer, 1, b, P + 1)).reshape(-1)

    codes, params = split_flat(flat.cpu().numpy(), 2, B, nkv, max_ctx, d)
    gpu_cache = oracle.Affine8Cache(codes.copy(), params.copy())
    appended_rows_valid(gpu_cache, ref_cache, init, min_exact=0.97)
    for b, P in enumerate(positions):
        # V is quantized from the same float32 inputs on both sides: bit-exact
        assert np.array_equal(gpu_cache.codes[layer, 1, b, :, P], ref_cache.codes[layer, 1, b, :, P])
        assert np.array_equal(gpu_cache.params[layer, 1, b, :, P], ref_cache.params[layer, 1, b, :, P])
        same_k = (np.array_equal(gpu_cache.codes[layer, 0, b, :, P], ref_cache.codes[layer, 0, b, :, P]) and
                  np.array_equal(gpu_cache.params[layer, 0, b, :, P], ref_cache.params[layer, 0, b, :, P]))
        err = np.abs(got[b] - ref[b])
        if same_k:
            assert np.all(err <= ATTN_ATOL + ATTN_RTOL * np.abs(ref[b])), f"seq {b}: max err {err.max():.3e}"
        else:  # a neighbouring code of the new key: the score of one position moves slightly
            assert np.all(err <= 2e-2), f"seq {b} (appended K on a rounding boundary): max err {err.max():.3e}"


# ------------------------------------------------------------------ whole steps

def _run_kv8(glue, wl, steps, graph=True, cache_weights=True, full_kv_check=True, plan=None):
    """Greedy loop on the GPU over an affine 8-bit cache, then the oracle replays the GPU's
    tokens; plan as in the bf16 step tests (default: every sequence over every step)."""
    model = synthetic.generate(wl, device="cuda")
    host = synthetic.to_host(model)
    init = host_cache(host["kv"])
    flat = synthetic.kv_buffer(model["kv"])
    dec = glue.Decoder(wl, model)
    dec.set_graph_mode(graph)
    try:
        assert dec.kv_cache_bytes == flat.numel()
        gpu_steps, _ = gpu_greedy(dec, dict(model, kv=flat), steps)
        st, bits = dec.device_status()
        assert bits == 0, f"device status bits {bits}"
    finally:
        dec.close()
    m = oracle.OracleModel.from_synthetic(wl, host, cache_weights=cache_weights)
    worst = {"max_abs": 0.0, "rel_l2": 0.0, "exempt": 0, "replayed": []}
    L, B, nkv, d = wl.n_layers, wl.batch, wl.n_kv_heads, wl.head_dim
    for seqs, n in plan or [(None, steps)]:
        res, ref_cache = oracle_replay(wl, host, init, gpu_steps[:n], seqs=seqs, model=m)
        sel = slice(None) if seqs is None else np.asarray(seqs)
        for s, lg, am in res:
            w = check_logits(gpu_steps[s][2][sel], lg, gpu_steps[s][3][sel], am,
                             f"{wl.name} step {s} seqs {'all' if seqs is None else list(seqs)}")
            worst["max_abs"] = max(worst["max_abs"], w["max_abs"])
            worst["rel_l2"] = max(worst["rel_l2"], w["rel_l2"])
            worst["exempt"] += w["exempt"]
        worst["replayed"].append(("all" if seqs is None else list(seqs), n))
        if full_kv_check and seqs is None and n == steps:
            codes, params = split_flat(flat.cpu().numpy(), L, B, nkv, wl.max_ctx, d)
            worst["rows_differ"] = appended_rows_valid(oracle.Affine8Cache(codes, params), ref_cache, init)
        else:  # only the appended slots (the full cache is several GB)
            nel = L * 2 * B * nkv * wl.max_ctx * d
            off = (nel + 255) // 256 * 256
            cv = flat[:nel].view(L, 2, B, nkv, wl.max_ctx, d)
            pv = flat[off: off + nel // 16].view(torch.int16).view(L, 2, B, nkv, wl.max_ctx, d // 64, 2)
            idx = range(B) if seqs is None else seqs
            for _, pin, _, _ in gpu_steps[:n]:
                for j, b in enumerate(idx):
                    P = int(pin[b])
                    g = oracle.Affine8Cache(cv[:, :, b:b + 1, :, P:P + 1].cpu().numpy().copy(),
                                            pv[:, :, b:b + 1, :, P:P + 1].cpu().numpy().view(np.uint16).copy())
                    r = oracle.Affine8Cache(ref_cache.codes[:, :, j:j + 1, :, P:P + 1].copy(),
                                            ref_cache.params[:, :, j:j + 1, :, P:P + 1].copy())
                    i0 = oracle.Affine8Cache(init.codes[:, :, b:b + 1, :, P:P + 1].copy(),
                                             init.params[:, :, b:b + 1, :, P:P + 1].copy())
                    appended_rows_valid(g, r, i0, min_exact=0.95)
    return worst


def test_kv8_tiny_all_steps(glue):
    w = _run_kv8(glue, synthetic.WORKLOADS["tiny-kv8"], 16)
    print("tiny-kv8 worst", w)


KV8_CUSTOM = [
    ("kv8_d128_g4_multi_split", dict(head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=256, intermediate=512,
                                     vocab=777, prefill=700, steps=3)),
    ("kv8_d64_g1_empty_cache", dict(head_dim=64, n_q_heads=2, n_kv_heads=2, hidden=128, intermediate=256,
                                    vocab=1003, prefill=0, steps=3)),
    ("kv8_b3_bf16_ragged", dict(batch=3, prefill=(0, 300), head_dim=128, n_q_heads=4, n_kv_heads=2, hidden=256,
                                intermediate=512, vocab=1000, steps=3, n_layers=2)),
    ("kv8_b12_q4_d64", dict(batch=12, weight_format=synthetic.AFFINE4_G64, prefill=(10, 600), head_dim=64,
                            n_q_heads=8, n_kv_heads=2, hidden=192, intermediate=384, vocab=517, steps=2,
                            n_layers=2)),
]


@pytest.mark.parametrize("name,kw", KV8_CUSTOM, ids=[c[0] for c in KV8_CUSTOM])
def test_kv8_custom_shapes(glue, name, kw):
    wl = synthetic.custom(name=name, seed=sum(map(ord, name)), kv_format=synthetic.AFFINE8_G64, **kw)
    assert wl.max_ctx % 16 == 0
    w = _run_kv8(glue, wl, wl.steps)
    print(name, w)


def test_kv8_graph_equals_eager_bitwise(glue):
    wl = synthetic.WORKLOADS["tiny-kv8"].replace(batch=3)
    outs = []
    for graph in (True, False):
        model = synthetic.generate(wl, device="cuda")
        dec = glue.Decoder(wl, model)
        dec.set_graph_mode(graph)
        steps, kv = gpu_greedy(dec, dict(model, kv=synthetic.kv_buffer(model["kv"])), 4)
        dec.close()
        outs.append((steps, kv.cpu()))
    for a, b in zip(outs[0][0], outs[1][0]):
        assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])
    assert torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("T,kw", [
    (4, dict(batch=2, head_dim=128, n_q_heads=4, n_kv_heads=2, hidden=256, intermediate=512, prefill=(60, 130),
             n_layers=2)),
    (3, dict(batch=3, weight_format=synthetic.AFFINE4_G64, head_dim=64, n_q_heads=4, n_kv_heads=1, hidden=256,
             intermediate=512, prefill=(0, 141), n_layers=2)),
])
def test_kv8_verify_matches_oracle(glue, T, kw):
    wl = synthetic.custom(name=f"kv8_verify_{T}", seed=40 + T, steps=T, kv_format=synthetic.AFFINE8_G64, **kw)
    assert wl.max_ctx % 16 == 0 and wl.max_ctx >= wl.max_prefill + T
    model = synthetic.generate(wl, device="cuda")
    host = synthetic.to_host(model)
    init = host_cache(host["kv"])
    flat = synthetic.kv_buffer(model["kv"])
    B, V = wl.batch, wl.vocab
    g = torch.Generator(device="cpu")
    g.manual_seed(17 * T)
    toks = torch.randint(0, V, (B, T), generator=g, dtype=torch.int32)
    dec = glue.Decoder(wl, model, tokens_per_seq=T)
    try:
        logits = torch.empty((B * T, V), dtype=torch.float32, device="cuda")
        argmax = torch.empty((B * T,), dtype=torch.int32, device="cuda")
        dec.step(toks.reshape(-1).cuda(), model["positions"], flat, logits, argmax)
        torch.cuda.synchronize()
        assert dec.device_status()[1] == 0
        lg = logits.cpu().numpy().reshape(B, T, V)
        am = argmax.cpu().numpy().reshape(B, T)
    finally:
        dec.close()
    m = oracle.OracleModel.from_synthetic(wl, host)
    ref_cache = init.copy()
    ref_lg, ref_am = oracle.verify_step(m, ref_cache, toks.numpy(), host["positions"].numpy())
    for t in range(T):
        check_logits(lg[:, t], ref_lg[:, t], am[:, t], ref_am[:, t], f"kv8 verify token {t}")
    codes, params = split_flat(flat.cpu().numpy(), wl.n_layers, B, wl.n_kv_heads, wl.max_ctx, wl.head_dim)
    appended_rows_valid(oracle.Affine8Cache(codes, params), ref_cache, init)


@pytest.mark.parametrize("name", ["qwen3-8b-b1-kv8", "qwen3-8b-q4-b32-kv8"])
def test_kv8_full_size_all_steps(glue, name):
    """Full-size kv8 workloads in the launch configuration the bench times, every greedy
    step against the oracle (batch 32: three fixed sequences over all steps, every sequence
    over the first two)."""
    wl = synthetic.WORKLOADS[name]
    w = _run_kv8(glue, wl, wl.steps, full_kv_check=False, plan=replay_plan(wl))
    print(name, "worst", w)

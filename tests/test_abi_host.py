"""CPU-only checks of the C-ABI library: it loads, exports every symbol that
include/dec.h declares, and rejects bad configurations on the host before any
CUDA call (so these run without a GPU)."""

import ctypes
import pathlib
import re
import subprocess

import pytest

ROOT = pathlib.Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "dec.h"


@pytest.fixture(scope="module")
def dec():
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import dec as d
    return d


def declared_functions():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"DEC_API\s+[\w\s\*]+?\b(dec_\w+)\s*\(", text)))


def test_header_declares_the_core_calls():
    names = declared_functions()
    for core in ("dec_create", "dec_step", "dec_destroy", "dec_kv_cache_bytes", "dec_last_error"):
        assert core in names


def test_library_exports_every_declared_symbol(dec):
    out = subprocess.run(["nm", "-D", "--defined-only", str(dec._LIB_PATH)], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (dec_\w+)", out))
    missing = set(declared_functions()) - exported
    assert not missing, f"declared but not exported: {missing}"
    for name in declared_functions():
        assert hasattr(dec.lib, name)


def _cfg(dec, **kw):
    base = dict(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, intermediate=768, vocab=4096,
                rms_eps=1e-6, rope_theta=1e6, linear_fmt=0, batch=1, max_ctx=144)
    base.update(kw)
    return dec.DecConfig(**base)


def test_kv_cache_bytes(dec):
    assert dec.dec_kv_cache_bytes(_cfg(dec)) == 2 * 2 * 1 * 2 * 144 * 64 * 2
    assert dec.lib.dec_kv_cache_bytes(None) == 0
    # affine 8-bit: the codes, padded to 256 bytes, then a (scale, bias) bf16 pair per 64
    codes = 2 * 2 * 3 * 2 * 144 * 128
    pad = (-codes) % 256
    assert dec.dec_kv_cache_bytes(_cfg(dec, kv_fmt=1, batch=3, head_dim=128)) == codes + pad + codes // 64 * 4
    codes = 2 * 2 * 1 * 2 * 144 * 64
    assert dec.dec_kv_cache_bytes(_cfg(dec, kv_fmt=1)) == codes + (-codes) % 256 + codes // 16
    assert dec.dec_kv_cache_bytes(_cfg(dec, kv_fmt=5)) == 0


def test_kv_cache_bytes_match_the_synthetic_buffer(dec):
    import synthetic
    from token_decode_step_gb300 import torch_glue
    wl = synthetic.WORKLOADS["tiny-kv8"].replace(batch=2)
    buf = synthetic.kv_buffer(synthetic.generate(wl)["kv"])
    assert dec.dec_kv_cache_bytes(torch_glue.make_config(wl)) == buf.numel()


def test_kv_quantize_rejects_bad_arguments(dec):
    with pytest.raises(dec.DecError) as ei:
        dec.dec_kv_quantize(0, 4, 96, 0, 0, 0)
    assert "head_dim" in str(ei.value)
    with pytest.raises(dec.DecError) as ei:
        dec.dec_kv_quantize(0, 4, 64, 0, 0, 0)
    assert "NULL" in str(ei.value)
    with pytest.raises(dec.DecError):
        dec.dec_kv_quantize(0, -1, 64, 0, 0, 0)
    dec.dec_kv_quantize(0, 0, 64, 0, 0, 0)  # nothing to quantize: no launch, no error


@pytest.mark.parametrize("kw,status,msg", [
    (dict(head_dim=96), 2, "head_dim"),
    (dict(n_q_heads=6, n_kv_heads=2), 2, "1, 2 or 4"),
    (dict(n_q_heads=5, n_kv_heads=2), 1, "multiple"),
    (dict(hidden=200), 2, "multiples of 64"),
    (dict(rms_eps=0.0), 1, "rms_eps"),
    (dict(linear_fmt=7), 1, "linear_fmt"),
    (dict(vocab=0), 1, "positive"),
    (dict(tokens_per_seq=4097), 2, "tokens_per_seq"),
    (dict(tokens_per_seq=-1), 1, "tokens_per_seq"),
    (dict(batch=20, tokens_per_seq=4096), 2, "rows"),
    (dict(kv_fmt=3), 1, "kv_fmt"),
    (dict(kv_fmt=1, max_ctx=150), 2, "multiple of 16"),
    (dict(proj_kernels=3), 1, "proj_kernels"),
    (dict(proj_kernels=-1), 1, "proj_kernels"),
])
def test_create_rejects_bad_config(dec, kw, status, msg):
    with pytest.raises(dec.DecError) as ei:
        dec.dec_create(_cfg(dec, **kw), dec.DecWeights())
    assert msg in str(ei.value)


def test_create_rejects_null_weights(dec):
    with pytest.raises(dec.DecError) as ei:
        dec.dec_create(_cfg(dec), dec.DecWeights())
    assert "non-NULL" in str(ei.value)


def test_create_rejects_misaligned_weight_pointer(dec):
    layers = (dec.DecLayerWeights * 2)()
    for i in range(2):
        lw = dec.DecLayerWeights(16, 16, 16, 16, *(dec.DecLinear(32, None, None) for _ in range(7)))
        layers[i] = lw
    layers[1].o = dec.DecLinear(40, None, None)  # not 16-byte aligned
    w = dec.DecWeights(16, 16, dec.DecLinear(16, None, None), ctypes.cast(layers, ctypes.POINTER(dec.DecLayerWeights)))
    with pytest.raises(dec.DecError) as ei:
        dec.dec_create(_cfg(dec), w)
    assert "layer 1 o" in str(ei.value)


def test_step_rejects_null_handle(dec):
    st = dec.lib.dec_step(None, 16, 16, 16, None, 16, None)
    assert st == dec.DEC_ERR_INVALID_ARG
    assert "handle" in dec.dec_last_error()


def test_force_timeout_rejects_bad_arguments(dec):
    assert dec.lib.dec_debug_force_timeout(None, 16, None) == dec.DEC_ERR_INVALID_ARG
    assert "polls" in dec.dec_last_error()


def test_step_host_rejects_null_handle(dec):
    st = dec.lib.dec_step_host(None, 16, 16, 16, None, 16, None)
    assert st == dec.DEC_ERR_INVALID_ARG
    assert "handle" in dec.dec_last_error()


@pytest.mark.parametrize("kw,msg", [
    (dict(logits=None), "NULL"),
    (dict(tokens=None), "NULL"),
    (dict(batch=0), "batch"),
    (dict(top_p=0.0), "top_p"),
    (dict(top_p=1.5), "top_p"),
    (dict(temperature=float("nan")), "temperature"),
])
def test_sample_rejects_bad_arguments(dec, kw, msg):
    args = dict(logits=16, batch=1, vocab=8, tokens=16, temperature=1.0, top_p=1.0)
    args.update(kw)
    prm = dec.SamplingParams(temperature=args["temperature"], top_k=0, top_p=args["top_p"], seed=1, offset=0,
                             offset_device=None)
    st = dec.lib.dec_sample(args["logits"], args["batch"], args["vocab"], prm, args["tokens"], None)
    assert st == dec.DEC_ERR_INVALID_ARG
    assert msg in dec.dec_last_error()


@pytest.mark.parametrize("entry", ["dec_attention", "dec_attention_noalloc"])
@pytest.mark.parametrize("kw,status,msg", [
    (dict(tokens_per_seq=2), 2, "tokens_per_seq"),
    (dict(kv_fmt=4), 1, "kv_fmt"),
    (dict(kv_fmt=1, max_ctx=150), 2, "multiple of 16"),
    (dict(head_dim=96), 2, "head_dim"),
    (dict(n_q_heads=5, n_kv_heads=2), 1, "multiple"),
])
def test_attention_entry_points_reject_the_same_configs(dec, entry, kw, status, msg):
    """dec_attention and dec_attention_noalloc share their config checks: a multi-token
    config (whose rows the stand-alone kernels would read as separate sequences) and the
    other unsupported shapes are refused by both, before any CUDA call."""
    cfg = _cfg(dec, **kw)
    if entry == "dec_attention":
        st = dec.lib.dec_attention(ctypes.byref(cfg), 0, 16, 16, 16, 16, 16, 16, 256, 1 << 20, None)
    else:
        st = dec.lib.dec_attention_noalloc(ctypes.byref(cfg), 0, 16, 16, 16, 16, 16, 16, None)
    assert st == status
    assert msg in dec.dec_last_error()


def test_btc_schedule_segments(dec):
    """Host side of the stream-K deal: the partial slots it asks for cover every tile's
    segments (checked against a direct count of the CTA ranges)."""
    for N, K, ctas in [(24576, 4096, 152), (4096, 12288, 152), (6144, 4096, 152), (128, 64, 152), (1000, 2560, 5)]:
        tiles, kst = (N + 127) // 128, K // 64
        total = tiles * kst
        grid = min(total, ctas)
        begin = [c * total // grid for c in range(grid + 1)]
        most = 1
        for t in range(tiles):
            owners = {c for c in range(grid) if begin[c] < (t + 1) * kst and begin[c + 1] > t * kst}
            most = max(most, len(owners))
        assert dec.lib.dec_debug_btc_max_segments(N, K, ctas) == most


def test_projection_plan(dec):
    """Host side of dec_config.proj_kernels: which projections run on the tcgen05 decode kernels
    (bit i: 0 q/k/v, 1 o, 2 gate/up, 3 down, 4 lm_head).  AUTO puts the gate/up and lm_head
    projections of 4-bit steps with 16..32 rows at hidden >= 2048 there; TCGEN05 every projection
    of 2..32-row steps at hidden >= 2048; batch-1, bf16-under-AUTO, small-hidden and 33+-row steps
    none."""
    big = dict(n_layers=1, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128, intermediate=12288,
               vocab=151936, max_ctx=64)
    GU_LM, ALL = 4 | 16, 31
    cases = [
        (dict(linear_fmt=1, batch=32, proj_kernels=0), GU_LM),
        (dict(linear_fmt=1, batch=32, proj_kernels=1), 0),
        (dict(linear_fmt=1, batch=32, proj_kernels=2), ALL),
        (dict(linear_fmt=1, batch=16, proj_kernels=0), GU_LM),
        (dict(linear_fmt=1, batch=15, proj_kernels=0), 0),
        (dict(linear_fmt=1, batch=8, proj_kernels=2), ALL),
        (dict(linear_fmt=1, batch=2, tokens_per_seq=8, proj_kernels=0), GU_LM),  # a 16-row verify step
        (dict(linear_fmt=1, batch=33, proj_kernels=2), 0),
        (dict(linear_fmt=1, batch=1, proj_kernels=2), 0),
        (dict(linear_fmt=0, batch=8, proj_kernels=0), 0),
        (dict(linear_fmt=0, batch=8, proj_kernels=2), ALL),
        (dict(linear_fmt=0, batch=1, tokens_per_seq=512, proj_kernels=2), 0),  # a prefill chunk
        (dict(linear_fmt=1, batch=32, proj_kernels=2, hidden=1024, n_q_heads=16, intermediate=3072), 0),
    ]
    for kw, want in cases:
        cfg = _cfg(dec, **{**big, **kw})
        assert dec.dec_debug_proj_plan(cfg) == want, kw
    mask = ctypes.c_int(-1)
    assert dec.lib.dec_debug_proj_plan(None, ctypes.byref(mask)) == dec.DEC_ERR_INVALID_ARG
    bad = _cfg(dec, **{**big, "proj_kernels": 3})
    assert dec.lib.dec_debug_proj_plan(ctypes.byref(bad), ctypes.byref(mask)) == dec.DEC_ERR_INVALID_ARG
    assert mask.value == -1


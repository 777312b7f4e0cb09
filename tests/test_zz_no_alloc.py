"""The allocation-free attention entry point (dec_attention_noalloc) against the
workspace entry point (dec_attention), through the C ABI, on two calls in a row.

dec_attention_noalloc serves callers that cannot allocate device memory when
they call it (for example while a stream is captured in global mode, or in a
host that hands over only input and output buffers); its scratch is a fixed
array inside the library.  This file is collected last on purpose, so a run that
stops at the first failure has already run every other test; it must also pass
when run alone in a fresh process.
"""

import pytest
import torch

from parity import attention_cfg, make_attention_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import dec as d
    return d


def _kv8_cache(seed, B, nkv, d, max_ctx, L=2):
    """A flat affine 8-bit cache buffer (codes, then (scale, bias) pairs) with the synthetic
    recipe's stored form."""
    import synthetic
    wl = synthetic.custom(name="noalloc", seed=seed, n_layers=L, n_kv_heads=nkv, n_q_heads=nkv, head_dim=d,
                          batch=B, prefill=max_ctx - 1, steps=1, kv_format=synthetic.AFFINE8_G64)
    assert wl.max_ctx == max_ctx
    return synthetic.kv_buffer(synthetic.generate(wl, device="cuda")["kv"])


@pytest.mark.parametrize("kv_fmt", [0, 1], ids=["bf16_cache", "affine8_cache"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(dec, kv_fmt):
    """Both entry points run the same kernels on the same inputs: outputs and the appended
    K/V must be identical bit for bit, on a first call and on a second call that appends the
    next position (the fixed array then holds the first call's table)."""
    B, nq, nkv, d, max_ctx = 3, 16, 4, 128, 2112
    positions = [1500, 37, 0]
    qkv, q_norm, k_norm, kv, pos = make_attention_case(77, B, nq, nkv, d, positions, max_ctx)
    cfg = attention_cfg(dec, B, nq, nkv, d, max_ctx)
    cfg.kv_fmt = kv_fmt
    if kv_fmt == 1:
        kv = _kv8_cache(78, B, nkv, d, max_ctx)
        assert kv.numel() == dec.dec_kv_cache_bytes(cfg)
    ws = torch.empty((dec.dec_attention_workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    d_qkv, d_qn, d_kn, d_pos = (t.cuda() for t in (qkv, q_norm, k_norm, pos))
    kv_a, kv_b = kv.cuda().clone(), kv.cuda().clone()
    s = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        # the second call appends the next position of every sequence
        d_pos.copy_(pos + call)
        out_a = torch.full((B, nq * d), float("nan"), device="cuda")
        out_b = torch.full((B, nq * d), float("nan"), device="cuda")
        dec.dec_attention(cfg, 1, d_qkv.data_ptr(), d_qn.data_ptr(), d_kn.data_ptr(), d_pos.data_ptr(),
                          kv_a.data_ptr(), out_a.data_ptr(), ws.data_ptr(), ws.numel(), s)
        dec.dec_attention_noalloc(cfg, 1, d_qkv.data_ptr(), d_qn.data_ptr(), d_kn.data_ptr(), d_pos.data_ptr(),
                                  kv_b.data_ptr(), out_b.data_ptr(), s)
        torch.cuda.synchronize()
        assert torch.isfinite(out_b).all(), f"call {call}"
        assert torch.equal(out_a, out_b), f"call {call}: outputs differ"
        assert torch.equal(kv_a, kv_b), f"call {call}: appended K/V differ"


def test_noalloc_rejects_shapes_beyond_its_scratch(dec):
    cfg = attention_cfg(dec, 4096, 32, 8, 128, 64)  # RoPE table of 4096 sequences > 1 MiB
    x = torch.zeros((16,), device="cuda")
    with pytest.raises(dec.DecError) as ei:
        dec.dec_attention_noalloc(cfg, 0, x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                  x.data_ptr(), 0)
    assert ei.value.status == dec.DEC_ERR_UNSUPPORTED
    assert "scratch" in str(ei.value)

"""Kernel-level GPU parity: the fused attention kernel (dec_attention, the kernel
dec_step runs for each layer) against the oracle's own sub-functions, on ragged
batches, empty caches and contexts that span many splits and tiles."""

import numpy as np
import pytest
import torch

import oracle
from oracle import numerics

from parity import ATTN_ATOL as ATOL, ATTN_RTOL as RTOL, attention_cfg, kv_appended_close, make_attention_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import dec as d
    return d


def oracle_attention(qkv, q_norm, k_norm, kv_bits, positions, layer, nq, nkv, d, eps, theta):
    """The attention part of the oracle's decode step for one layer; writes the
    appended slots into kv_bits (numpy uint16) and returns out [B, nq*d]."""
    B = qkv.shape[0]
    qn = numerics.bf16_bits_to_f64(q_norm)
    kn = numerics.bf16_bits_to_f64(k_norm)
    out = np.empty((B, nq * d))
    for b in range(B):
        P = int(positions[b])
        q = oracle.rmsnorm(qkv[b, : nq * d].reshape(nq, d), qn, eps)
        k = oracle.rmsnorm(qkv[b, nq * d:(nq + nkv) * d].reshape(nkv, d), kn, eps)
        v = qkv[b, (nq + nkv) * d:].reshape(nkv, d)
        q = oracle.rope_rotate_half(q, P, theta)
        k = oracle.rope_rotate_half(k, P, theta)
        kv_bits[layer, 0, b, :, P, :] = numerics.f64_to_bf16_bits(k)
        kv_bits[layer, 1, b, :, P, :] = numerics.f64_to_bf16_bits(v)
        K = numerics.bf16_bits_to_f64(kv_bits[layer, 0, b, :, : P + 1, :])
        V = numerics.bf16_bits_to_f64(kv_bits[layer, 1, b, :, : P + 1, :])
        out[b] = oracle.gqa_attention(q, K, V).reshape(-1)
    return out


CASES = [
    # B, nq, nkv, d, positions, max_ctx
    (1, 16, 8, 128, [1024], 1152),
    (3, 8, 2, 64, [0, 65, 700], 800),
    (2, 32, 8, 128, [4095, 513], 4160),
    (4, 4, 4, 128, [2000, 1, 64, 127], 2080),
    (2, 8, 4, 64, [8191, 3], 8224),
    # more (sequence, KV head) pairs than fit one CTA per SM in clusters of 8: the
    # shallow two-CTAs-per-SM ring
    (6, 16, 4, 128, [1500, 0, 63, 64, 777, 1200], 1536),
    (12, 4, 2, 64, [5, 300, 17, 1000, 64, 129, 2, 999, 640, 31, 1023, 256], 1024),
    # clusters of 8 would take two waves of two CTAs per SM, clusters of 4 take one
    (10, 16, 4, 128, [900, 1, 2047, 333, 64, 65, 1500, 0, 1000, 2000], 2048),
    # the batch-32 8B shapes: 256 clusters of 4, several waves of two CTAs per SM
    (32, 32, 8, 128, [int(x) for x in np.random.default_rng(32).integers(512, 8193, 32)], 8224),
]


def run_kernel(dec, cfg, layer, qkv, q_norm, k_norm, pos, kv, out, workspace):
    s = torch.cuda.current_stream().cuda_stream
    dec.dec_attention(cfg, layer, qkv.data_ptr(), q_norm.data_ptr(), k_norm.data_ptr(), pos.data_ptr(),
                      kv.data_ptr(), out.data_ptr(), workspace.data_ptr(), workspace.numel(), s)


@pytest.mark.parametrize("B,nq,nkv,d,positions,max_ctx", CASES)
def test_attention_kernel_matches_oracle(dec, B, nq, nkv, d, positions, max_ctx):
    qkv, q_norm, k_norm, kv, pos = make_attention_case(B * 100 + d, B, nq, nkv, d, positions, max_ctx)
    cfg = attention_cfg(dec, B, nq, nkv, d, max_ctx)
    ws_bytes = dec.dec_attention_workspace_bytes(cfg)
    assert ws_bytes > 0
    workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device="cuda")
    workspace.fill_(0xAB)  # contents on entry must not matter
    kv_bits0 = kv.view(torch.int16).numpy().view(np.uint16).copy()
    d_qkv, d_qn, d_kn, d_kv, d_pos = (t.cuda() for t in (qkv, q_norm, k_norm, kv, pos))
    out = torch.full((B, nq * d), float("nan"), device="cuda")
    layer = 1
    run_kernel(dec, cfg, layer, d_qkv, d_qn, d_kn, d_pos, d_kv, out, workspace)
    torch.cuda.synchronize()
    kv_ref = kv_bits0.copy()
    ref = oracle_attention(qkv.double().numpy(), q_norm.view(torch.int16).numpy().view(np.uint16),
                           k_norm.view(torch.int16).numpy().view(np.uint16), kv_ref, positions, layer, nq, nkv, d,
                           1e-6, 1e6)
    got = out.cpu().double().numpy()
    err = np.abs(got - ref)
    assert np.all(err <= ATOL + RTOL * np.abs(ref)), f"max err {err.max():.3e}"
    kv_gpu = d_kv.cpu().view(torch.int16).numpy().view(np.uint16)
    # everything but the appended slots untouched; appended vectors within 2 bf16 steps
    kv_appended_close(kv_gpu, kv_ref, kv_bits0)
    for b, P in enumerate(positions):
        assert np.any(kv_gpu[layer, :, b, :, P, :] != kv_bits0[layer, :, b, :, P, :])


def test_attention_rejects_small_workspace(dec):
    cfg = attention_cfg(dec, 1, 4, 2, 64, 100)
    need = dec.dec_attention_workspace_bytes(cfg)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 8 * 64), device="cuda")
    with pytest.raises(dec.DecError):
        dec.dec_attention(cfg, 0, x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                          x.data_ptr(), ws.data_ptr(), need - 256, 0)

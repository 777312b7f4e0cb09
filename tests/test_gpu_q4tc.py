"""The batched-decode projection kernel for affine 4-bit weights on tcgen05
(dec_debug_gemm_q4tc, plain store epilogue) against an fp64 product of the same inputs, the
weights dequantized by the oracle (fl(scale * q + bias), float32): ragged token counts and
weight-row tiles, K splits, more groups than the stage rings hold; and the bf16 form."""

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import dec as d
    return d


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K,S", [(32, 128, 64, 1), (32, 256, 1024, 2), (8, 200, 512, 1), (17, 1000, 2560, 5),
                                     (1, 130, 384, 3), (32, 6144, 4096, 8), (32, 4096, 12288, 4),
                                     # odd groups per split: the last two-group stage of each unit holds one
                                     (32, 250, 320, 1), (8, 300, 2560, 8), (5, 977, 1344, 3)])
def test_q4tc_gemm_matches_fp64(dec, M, N, K, S):
    g = torch.Generator(device="cpu")
    g.manual_seed(M * 7 + N + K + S)
    x = torch.randn((M, K), generator=g, dtype=torch.float64)
    hi = x.to(torch.bfloat16)
    lo = (x - hi.double()).to(torch.bfloat16)
    words = torch.randint(-(2 ** 31), 2 ** 31, (N, K // 8), generator=g, dtype=torch.int64).to(torch.int32)
    scales = _bf16_bits(torch.rand((N, K // 64), generator=g) * 0.009 + 0.001)
    biases = _bf16_bits(torch.randn((N, K // 64), generator=g) * 0.02)
    w = oracle.dequant_affine4_g64_f32(words.numpy().view(np.uint32), scales, biases).astype(np.float64)
    sb = scales.astype(np.uint32) | (biases.astype(np.uint32) << 16)

    xhl = torch.stack([hi, lo]).contiguous().cuda()
    wd = words.contiguous().cuda()
    sbd = torch.from_numpy(sb.view(np.int32)).contiguous().cuda()
    out = torch.full((M, N), float("nan"), device="cuda")
    partials = torch.empty((S, M, N), device="cuda") if S > 1 else None
    counters = torch.zeros(((N + 119) // 120 + 1,), dtype=torch.int32, device="cuda") if S > 1 else None
    dec.dec_debug_gemm_q4tc(xhl.data_ptr(), M, wd.data_ptr(), sbd.data_ptr(), N, K, S, out.data_ptr(),
                            partials.data_ptr() if S > 1 else None, counters.data_ptr() if S > 1 else None,
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    xs = (hi.double() + lo.double()).numpy()
    ref = xs @ w.T
    bound = np.abs(xs) @ np.abs(w).T  # the products' magnitudes (x's hi/lo split keeps ~16 bits)
    got = out.cpu().double().numpy()
    assert np.isfinite(got).all(), "unwritten outputs"
    err = np.abs(got - ref)
    assert np.all(err <= 4e-5 * bound + 1e-6), f"max err {float(err.max()):.3e} (rel {float((err / bound).max()):.3e})"
    if S > 1:
        assert int(counters.abs().sum()) == 0, "split counters not left zero"


@pytest.mark.parametrize("M,N,K,ctas", [(8, 128, 64, 0), (8, 24576, 4096, 0), (16, 200, 512, 0), (32, 1000, 2560, 5),
                                        (3, 130, 384, 3), (8, 4096, 12288, 0), (8, 6144, 4096, 7), (17, 300, 1024, 1)])
def test_btc_gemm_matches_fp64(dec, M, N, K, ctas):
    """The bf16 form (dec_debug_gemm_btc): weights streamed by TMA into the MMA, the tiles' stages
    dealt stream-K to `ctas` CTAs (0: one per SM), so tiles split over several CTAs and their
    segments added through the partial slots."""
    g = torch.Generator(device="cpu")
    g.manual_seed(M * 11 + N + K + ctas)
    x = torch.randn((M, K), generator=g, dtype=torch.float64)
    hi = x.to(torch.bfloat16)
    lo = (x - hi.double()).to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g) * 0.05).to(torch.bfloat16)
    xhl = torch.stack([hi, lo]).contiguous().cuda()
    wd = w.contiguous().cuda()
    out = torch.full((M, N), float("nan"), device="cuda")
    partials = torch.empty((K // 64, M, N), device="cuda")
    counters = torch.zeros(((N + 127) // 128 + 1,), dtype=torch.int32, device="cuda")
    dec.dec_debug_gemm_btc(xhl.data_ptr(), M, wd.data_ptr(), N, K, ctas, out.data_ptr(), partials.data_ptr(),
                           counters.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    xs = (hi.double() + lo.double()).numpy()
    wf = w.double().numpy()
    ref = xs @ wf.T
    bound = np.abs(xs) @ np.abs(wf).T
    got = out.cpu().double().numpy()
    assert np.isfinite(got).all(), "unwritten outputs"
    err = np.abs(got - ref)
    assert np.all(err <= 1e-5 * bound + 1e-6), f"max err {float(err.max()):.3e}"
    assert int(counters.abs().sum()) == 0, "tile counters not left zero"


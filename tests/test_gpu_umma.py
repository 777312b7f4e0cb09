"""The prefill projection kernel on tcgen05 (dec_debug_gemm_tc5, plain store epilogue)
against an fp64 matrix product of the same bf16 inputs: ragged token and weight-row
tiles, more inputs than the stage ring holds."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_decode_step_gb300 import build
    build.build()
    from token_decode_step_gb300 import dec as d
    return d


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (300, 200, 320), (77, 384, 1024), (1000, 130, 256),
                                   # grids of one CTA per SM or more take 256-row weight tiles (ragged N here)
                                   (2048, 2600, 192), (1100, 5000, 128)])
@pytest.mark.parametrize("persistent", [0, 1])
def test_tc5_gemm_matches_fp64(dec, M, N, K, persistent):
    g = torch.Generator(device="cpu")
    g.manual_seed(M + N + K)
    x = torch.randn((M, K), generator=g, dtype=torch.float64)
    hi = x.to(torch.bfloat16)
    lo = (x - hi.double()).to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g) * 0.05).to(torch.bfloat16)
    xhl = torch.stack([hi, lo]).contiguous().cuda()
    wd = w.contiguous().cuda()
    out = torch.full((M, N), float("nan"), device="cuda")
    dec.dec_debug_gemm_tc5(xhl.data_ptr(), M, wd.data_ptr(), N, K, out.data_ptr(), persistent,
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref = (hi.double() + lo.double()) @ w.double().T
    got = out.cpu().double()
    err = (got - ref).abs()
    assert torch.isfinite(got).all(), "unwritten outputs"
    assert float(err.max()) <= 1e-5 * float(ref.abs().max()) + 1e-6, f"max err {float(err.max()):.3e}"

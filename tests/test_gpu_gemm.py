"""GPU check of the tcgen05 projection GEMM against float64 matmul."""

import numpy as np
import pytest
import torch

import differential_attention_02_gb300 as da
from parity import assert_bf16_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from differential_attention_02_gb300 import build
    build.build()
    da.load_library()


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 128), (200, 264, 72), (1, 8, 8), (1000, 2048, 2048)])
def test_gemm_against_float64(M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(K, N, generator=g) / K ** 0.5).to(torch.bfloat16)
    ref = a.double().numpy() @ w.double().numpy()
    ws = da.workspace(256)
    out = da.gemm_bf16(a.cuda(), w.cuda(), out_dtype=torch.float32, ws=ws)
    assert da.read_error(ws) == 0
    assert_bf16_parity(out, ref, f"gemm {M}x{N}x{K}")
    outb = da.gemm_bf16(a.cuda(), w.cuda(), out_dtype=torch.bfloat16, ws=ws)
    d = np.abs(outb.float().cpu().numpy() - ref)
    assert np.max(d - 2.0 ** -8 * np.abs(ref)) <= 1e-3


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 264, 72), (1000, 2048, 2048)])
def test_gemm_f16_operands(M, N, K):
    g = torch.Generator().manual_seed(M * 3 + N + K)
    a = torch.randn(M, K, generator=g).half()
    w = (torch.randn(K, N, generator=g) / K ** 0.5).half()
    ref = a.double().numpy() @ w.double().numpy()
    ws = da.workspace(256)
    out = da.gemm(a.cuda(), w.cuda(), out_dtype=torch.float32, ws=ws)
    assert da.read_error(ws) == 0
    # Exact fp16 products, fp32 accumulation over K: a few fp32 ulps of the partial sums.
    assert np.max(np.abs(out.cpu().double().numpy() - ref)) <= 1e-4 * max(1.0, K ** 0.5 / 8)
    with pytest.raises(ValueError):
        da.gemm(a.cuda(), w.cuda().to(torch.bfloat16))


def test_gemm_f16_output():
    g = torch.Generator().manual_seed(3)
    a = torch.randn(300, 512, generator=g).to(torch.bfloat16)
    w = (torch.randn(512, 384, generator=g) / 512 ** 0.5).to(torch.bfloat16)
    ref = a.double().numpy() @ w.double().numpy()
    out = da.gemm_bf16(a.cuda(), w.cuda(), out_dtype=torch.float16)
    assert out.dtype == torch.float16
    d = np.abs(out.double().cpu().numpy() - ref)
    assert np.max(d - 2.0 ** -11 * np.abs(ref)) <= 1e-3

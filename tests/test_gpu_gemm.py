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


# More tiles than SMs, so the persistent CTAs take a second round: (2500, 2048): 160 tiles of
# 128 x 256 with ragged last rows; (2304, 2112): 162 tiles, the last tile column partial;
# (3968, 2048): 248 tiles.
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 128), (200, 264, 72), (1, 8, 8), (1000, 2048, 2048),
                                   (2500, 2048, 512), (2304, 2112, 256), (3968, 2048, 256)])
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


# ------------------------------------------------------------- epilogue modes of the layer
def _fp32_accum_bar(ref, K):
    """fp32 accumulation over K exact 16-bit products: a few fp32 ulps of the partial sums."""
    return 1e-4 * max(1.0, K ** 0.5 / 8) * max(1.0, float(np.abs(ref).max()))


@pytest.mark.parametrize("M,N,K,r_dtype", [(200, 512, 72, torch.float32), (1, 256, 8, torch.bfloat16),
                                           (1000, 2048, 512, torch.float16), (384, 768, 2048, torch.float32),
                                           (2500, 2048, 256, torch.float16)])
def test_gemm_residual_against_float64(M, N, K, r_dtype):
    """C = A W + R (fp32), its 16-bit copy C * gain (fp16 and bf16) and the per-256-column row
    sums of C^2, each against float64 on the same inputs (the last case has more tiles than
    SMs)."""
    g = torch.Generator().manual_seed(M + 7 * N + K)
    a = torch.randn(M, K, generator=g).half()
    w = (torch.randn(K, N, generator=g) / K ** 0.5).half()
    r = (torch.randn(M, N, generator=g) * 3).to(r_dtype)
    gain = torch.linspace(0.5, 1.5, N)
    c64 = a.double().numpy() @ w.double().numpy() + r.double().numpy()
    ws = da.workspace(256)
    for c16_dtype in (torch.float16, torch.bfloat16):
        c, c16, sq = da.gemm_residual(a.cuda(), w.cuda(), r.cuda(), c16_dtype=c16_dtype, c16_gain=gain.cuda(),
                                      want_row_sq=True, ws=ws)
        torch.cuda.synchronize()
        assert da.read_error(ws) == 0
        got = c.cpu().double().numpy()
        assert np.max(np.abs(got - c64)) <= _fp32_accum_bar(c64, K)
        # the copy is the kernel's own fp32 C times the gain, rounded once (half an ulp)
        want16 = (c.cpu() * gain).to(c16_dtype)
        assert torch.equal(c16.cpu().view(torch.int16), want16.view(torch.int16)), c16_dtype
        sq64 = (c64 ** 2).reshape(M, N // 256, 256).sum(axis=2)
        np.testing.assert_allclose(sq.cpu().double().numpy(), sq64, rtol=1e-4 * max(1.0, K ** 0.5 / 8))
    # without the optional outputs
    c, c16, sq = da.gemm_residual(a.cuda(), w.cuda(), r.cuda(), ws=ws)
    assert c16 is None and sq is None
    assert np.max(np.abs(c.cpu().double().numpy() - c64)) <= _fp32_accum_bar(c64, K)


def _silu64(t):
    return t / (1.0 + np.exp(-t))


@pytest.mark.parametrize("M,F,K,with_sq", [(200, 256, 72, True), (1, 128, 8, False), (1000, 1536, 512, True)])
def test_gemm_swiglu_against_float64(M, F, K, with_sq):
    """H = SiLU(g / r) (u / r) from the interleaved gate/up weight, against float64 on the
    same 16-bit inputs (the fp32 GEMM error of g and u, then H's rounding to fp16)."""
    g0 = torch.Generator().manual_seed(M + F + K)
    a = torch.randn(M, K, generator=g0).half()
    wg = (torch.randn(K, F, generator=g0) / K ** 0.5).half()
    wu = (torch.randn(K, F, generator=g0) / K ** 0.5).half()
    sq = (torch.rand(M, 3, generator=g0) * 50 + 1) if with_sq else None
    w_gu = da.interleave_gate_up(wg, wu)
    # the interleaved layout: 128-column blocks of gate and up alternate
    assert torch.equal(w_gu[:, 128:256], wu[:, :128]) and torch.equal(w_gu[:, 256:384], wg[:, 128:256]) or F == 128
    a64 = a.double().numpy()
    gg, uu = a64 @ wg.double().numpy(), a64 @ wu.double().numpy()
    if with_sq:
        ir = 1.0 / np.sqrt(sq.double().numpy().sum(axis=1, keepdims=True) / 384.0 + 1e-5)
        gg, uu = gg * ir, uu * ir
    ref = _silu64(gg) * uu
    ws = da.workspace(256)
    h = da.gemm_swiglu(a.cuda(), w_gu.cuda(), row_sq=None if sq is None else sq.cuda(), sq_count=384.0, eps=1e-5,
                       out_dtype=torch.float16, ws=ws)
    torch.cuda.synchronize()
    assert da.read_error(ws) == 0 and h.shape == (M, F)
    d = np.abs(h.cpu().double().numpy() - ref)
    # fp16 rounding of H (2^-11 relative) plus the fp32 GEMM error carried through SiLU(g) u
    assert np.max(d - 2.0 ** -11 * np.abs(ref)) <= 2e-4 * max(1.0, float(np.abs(ref).max()))
    hb = da.gemm_swiglu(a.cuda(), w_gu.cuda(), row_sq=None if sq is None else sq.cuda(), sq_count=384.0, eps=1e-5,
                        out_dtype=torch.bfloat16, ws=ws)
    db = np.abs(hb.cpu().double().numpy() - ref)
    assert np.max(db - 2.0 ** -8 * np.abs(ref)) <= 2e-4 * max(1.0, float(np.abs(ref).max()))

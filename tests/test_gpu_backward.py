"""GPU parity of the backward pass (diffattn_bwd) against the float64 oracle's chain
rule of the definition, on seeded inputs.

Tolerance: the kernels compute in fp32 from inputs that the oracle sees exactly
(bf16 and fp16 values are exact in fp32), so the bar is fp32 accumulation error:
relative RMS <= 2e-5 per gradient tensor and max-abs <= 2e-4 of the tensor's
largest magnitude; dlambda and dw (sums over every row) within 1e-4 relative.
Rounding error scales with the terms that cancel, not with the result: a
gradient that the mathematics makes zero (a row with one visible key has
dS = P (dA - dA) = 0, so dQ = 0; the oracle's float64 value is ~1e-17) is checked
in absolute terms instead, max-abs <= 1e-5 of the largest gradient magnitude of
the call.
"""

import numpy as np
import pytest
import torch

import differential_attention_02_gb300 as da
from differential_attention_02_gb300 import inputs as gi
from oracle import diffattn_oracle as orc

pytestmark = pytest.mark.gpu
NAMES = ("q1", "q2", "k1", "k2", "v")
GRADS = ("dq1", "dq2", "dk1", "dk2", "dv")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from differential_attention_02_gb300 import build
    build.build()
    da.load_library()


def _check(g, ref, what, heads=None):
    pick = lambda a: a if heads is None else np.stack([a[b, h] for b, h in heads])
    scale = max(np.abs(pick(ref[k])).max() for k in GRADS)
    for k in GRADS:
        got = pick(g[k].cpu().double().numpy())
        exp = pick(ref[k])
        err = got - exp
        assert np.all(np.isfinite(got)), f"{what} {k}: non-finite"
        if np.abs(exp).max() <= 1e-9 * scale:  # zero by the mathematics
            ma = np.abs(err).max() / scale
            print(f"{what} {k}: zero gradient, max-abs/scale {ma:.2e}")
            assert ma <= 1e-5, f"{what} {k}: max-abs/scale {ma:.3e}"
            continue
        rr = np.linalg.norm(err) / np.linalg.norm(exp)
        ma = np.abs(err).max() / np.abs(exp).max()
        print(f"{what} {k}: rel-RMS {rr:.2e}, max-abs/max {ma:.2e}")
        assert rr <= 2e-5 and ma <= 2e-4, f"{what} {k}: rel-RMS {rr:.3e}, max-abs/max {ma:.3e}"


def _run(t, dy, lam, lam_init, eps=1e-5, **kw):
    ws = da.workspace(da.bwd_workspace_bytes(*t["q1"].shape, t["v"].shape[-1]))
    g = da.diffattn_bwd(*(t[k].cuda() for k in NAMES), dy.cuda(), lam, lam_init, eps, ws=ws, **kw)
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("B,H,N,d,Dv,causal,dtype", [
    (1, 1, 1, 32, 64, True, torch.float32),
    (1, 2, 45, 32, 64, True, torch.float32),
    (2, 1, 70, 64, 128, False, torch.bfloat16),
    (1, 2, 33, 128, 256, True, torch.float16),
    (1, 3, 130, 64, 128, True, torch.bfloat16),
    (2, 2, 300, 128, 256, True, torch.bfloat16),
])
def test_backward_shapes(B, H, N, d, Dv, causal, dtype):
    g0 = torch.Generator().manual_seed(B * 1000 + N * 7 + d)
    t = {k: torch.randn(B, H, N, Dv if k == "v" else d, generator=g0).to(dtype) for k in NAMES}
    dy = torch.randn(B, N, H, Dv, generator=g0).to(dtype)
    lam, lam_init = 0.58, 0.35
    g = _run(t, dy, lam, lam_init, causal=causal, want_dnorm_weight=True)
    ref = orc.diffattn_bwd(*(t[k] for k in NAMES), dy, lam, lam_init, 1e-5, causal=causal)
    _check(g, ref, f"B{B} H{H} N{N} d{d} {dtype}")
    assert float(g["dlam"].item()) == pytest.approx(ref["dlam"], rel=1e-4, abs=1e-6)
    np.testing.assert_allclose(g["dw"].cpu().double().numpy(), ref["dw"], rtol=1e-4, atol=1e-5)


@pytest.mark.parametrize("lam", [0.0, -0.8, 2.2])
def test_backward_lambda_values_and_norm_weight(lam):
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w, B=1, H=2, N=200)
    dy = gi.output_grad(w, B=1, H=2, N=200)
    nw = torch.linspace(0.5, 1.5, w.Dv)
    g = _run(t, dy, lam, 0.4, norm_weight=nw.cuda(), want_dnorm_weight=True)
    ref = orc.diffattn_bwd(*(t[k] for k in NAMES), dy, lam, 0.4, 1e-5, weight=nw.numpy())
    _check(g, ref, f"lambda {lam}")
    assert float(g["dlam"].item()) == pytest.approx(ref["dlam"], rel=1e-4, abs=1e-6)
    np.testing.assert_allclose(g["dw"].cpu().double().numpy(), ref["dw"], rtol=1e-4, atol=1e-5)
    if lam == 0.0:
        assert float(g["dq2"].abs().max()) == 0.0 and float(g["dk2"].abs().max()) == 0.0


def test_backward_strided_views():
    """Q1/Q2 and K1/K2 as halves of one [B, N, H, 2d] buffer, as the module lays them out."""
    B, H, N, d = 1, 2, 96, 64
    g0 = torch.Generator().manual_seed(9)
    qk = torch.randn(2, B, N, H, 2 * d, generator=g0).to(torch.bfloat16)
    v = torch.randn(B, N, H, 128, generator=g0).to(torch.bfloat16)
    dy = torch.randn(B, N, H, 128, generator=g0).to(torch.bfloat16)
    q4, k4 = qk[0].permute(0, 2, 1, 3), qk[1].permute(0, 2, 1, 3)
    t = {"q1": q4[..., :d], "q2": q4[..., d:], "k1": k4[..., :d], "k2": k4[..., d:], "v": v.permute(0, 2, 1, 3)}
    ref = orc.diffattn_bwd(*(t[k] for k in NAMES), dy, 0.5, 0.2)
    qkd, vd = qk.cuda(), v.cuda()
    q4d, k4d = qkd[0].permute(0, 2, 1, 3), qkd[1].permute(0, 2, 1, 3)
    g = da.diffattn_bwd(q4d[..., :d], q4d[..., d:], k4d[..., :d], k4d[..., d:], vd.permute(0, 2, 1, 3), dy.cuda(),
                        0.5, 0.2)
    torch.cuda.synchronize()
    _check(g, ref, "strided")


def test_backward_is_deterministic():
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w, B=1, H=2, N=257)
    dy = gi.output_grad(w, B=1, H=2, N=257)
    a = _run(t, dy, 0.5, 0.3, want_dnorm_weight=True)
    a = {k: v.clone() for k, v in a.items()}
    b = _run(t, dy, 0.5, 0.3, want_dnorm_weight=True)
    for k in GRADS + ("dlam", "dw"):
        assert torch.equal(a[k], b[k]), k


def test_backward_prefill_workload_sampled_heads():
    """The B=4, H=16, N=2048 prefill workload: every gradient of three heads, and dlambda, dw
    over all 64 heads."""
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w)
    dy = gi.output_grad(w)
    lv = gi.lambda_vectors(w)
    lam, lam_init = orc.reparam_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer)
    g = _run(t, dy, lam, lam_init, want_dnorm_weight=True)
    heads = [(0, 0), (1, 7), (3, 15)]
    ref = orc.diffattn_bwd(*(t[k] for k in NAMES), dy, lam, lam_init, w.eps)
    _check(g, ref, "prefill workload", heads=heads)
    assert float(g["dlam"].item()) == pytest.approx(ref["dlam"], rel=1e-4)
    np.testing.assert_allclose(g["dw"].cpu().double().numpy(), ref["dw"], rtol=1e-4, atol=1e-4)

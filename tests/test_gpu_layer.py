"""GPU parity of the DIFF Transformer layer (pre-RMSNorm, the differential
attention module, residual add, SwiGLU feed-forward, residual add) and of its
two elementwise kernels, against the float64 oracle."""

import numpy as np
import pytest
import torch

import differential_attention_02_gb300 as da
from differential_attention_02_gb300 import inputs as gi
from oracle import diffattn_oracle as orc
from parity import assert_bf16_out_parity, assert_bf16_parity, assert_f32_parity, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from differential_attention_02_gb300 import build
    build.build()
    da.load_library()


def _lam(w):
    lv = gi.lambda_vectors(w)
    return orc.reparam_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer)


# ------------------------------------------------------------ add + RMSNorm
@pytest.mark.parametrize("M,N,x_f32,with_z,with_w", [(1, 8, False, False, False), (37, 520, False, True, True),
                                                     (300, 2048, True, True, False), (5, 4104, True, False, True)])
@pytest.mark.parametrize("n_dtype", [torch.bfloat16, torch.float16])
def test_add_rmsnorm(M, N, x_f32, with_z, with_w, n_dtype):
    g = torch.Generator().manual_seed(M * 31 + N)
    x = torch.randn(M, N, generator=g) * 1.7
    x = x if x_f32 else x.to(torch.bfloat16)
    z = torch.randn(M, N, generator=g) if with_z else None
    wt = 1 + 0.1 * torch.randn(N, generator=g) if with_w else None
    dev = lambda t: None if t is None else t.cuda()
    y, n = da.add_rmsnorm(x.cuda(), dev(z), dev(wt), eps=1e-5, want_y=True, n_dtype=n_dtype)
    ref_y = x.double().numpy() + (0 if z is None else z.double().numpy())
    assert_f32_parity(y, ref_y, "y = x + z")
    ref_n = orc.rmsnorm_rows(ref_y, 1e-5, None if wt is None else wt.numpy())
    assert n.dtype == n_dtype
    # fp32 arithmetic, then one rounding to the output type: half an ulp, at most 2^-8 |n| for
    # bf16 (8 significant bits) and 2^-11 |n| for fp16 (11).
    half_ulp = 2.0 ** -8 if n_dtype == torch.bfloat16 else 2.0 ** -11
    err = np.abs(n.double().cpu().numpy() - ref_n) - half_ulp * np.abs(ref_n)
    assert err.max() <= 2e-6 * np.abs(ref_n).max(), f"RMSNorm(y): {err.max():.3e}"


def test_add_rmsnorm_outputs_optional():
    x = torch.randn(4, 64).cuda()
    y, n = da.add_rmsnorm(x, want_y=True, want_n=False)
    assert n is None and torch.equal(y, x)
    y, n = da.add_rmsnorm(x[:0], want_y=True)
    assert y.numel() == 0 and n.numel() == 0


# ------------------------------------------------------------------ SwiGLU
@pytest.mark.parametrize("M,H", [(1, 8), (13, 1536), (257, 5632)])
@pytest.mark.parametrize("h_dtype", [torch.bfloat16, torch.float16])
def test_swiglu(M, H, h_dtype):
    g = torch.Generator().manual_seed(M + H)
    gu = (torch.randn(M, 2 * H, generator=g) * 2.5).half()
    h = da.swiglu(gu.cuda(), out_dtype=h_dtype)
    assert h.dtype == h_dtype
    gd = gu.double().numpy()
    ref = orc.silu(gd[:, :H]) * gd[:, H:]
    half_ulp = 2.0 ** -8 if h_dtype == torch.bfloat16 else 2.0 ** -11
    err = np.abs(h.double().cpu().numpy() - ref) - half_ulp * np.abs(ref)
    assert err.max() <= 1e-5 * max(1.0, np.abs(ref).max()), f"SwiGLU M={M} H={H}: {err.max():.3e}"


def test_swiglu_saturates_cleanly():
    # SiLU's tails: t e^{-t} overflow must give 0 for t -> -inf, and t itself for t -> +inf.
    gu = torch.tensor([[-60000.0, -20.0, 0.0, 20.0, 60000.0, 1.0, -1.0, 3.0] + [2.0] * 8], dtype=torch.half)
    h = da.swiglu(gu.cuda()).float().cpu().numpy()[0]
    gd = gu.double().numpy()[0]
    ref = orc.silu(gd[:8]) * gd[8:]
    np.testing.assert_allclose(h, ref, rtol=2 ** -8, atol=1e-30)


# ------------------------------------------------------------------- layer
def _layer(w, t, op_dtype=torch.float16, fused_qkv=True):
    """Runs the layer with every weight as op_dtype. fp16 copies of the bf16 weights are exact
    above 2^-14 in magnitude; the smaller values (about 0.3%) move by at most 2^-25, and the
    oracle sees the bf16 values."""
    lam, lam_init = _lam(w)
    dev = {k: (v.cuda().to(op_dtype) if k.startswith("w_") else v.cuda()) for k, v in t.items()}
    ws = da.workspace(256)
    wgu = da.interleave_gate_up(dev["w_gate"], dev["w_up"])
    wqkv = torch.cat([dev["w_q"], dev["w_k"], dev["w_v"]], dim=1).contiguous() if fused_qkv else None
    out = da.layer_fwd(dev["x"], dev["w_q"], dev["w_k"], dev["w_v"], dev["w_o"], wgu, dev["w_down"], w.H, lam,
                       lam_init, w.eps, norm1_weight=dev.get("norm1_w"), norm2_weight=dev.get("norm2_w"), ws=ws,
                       w_qkv=wqkv)
    torch.cuda.synchronize()
    assert da.read_error(ws) == 0
    assert out.dtype == torch.float32 and out.shape == t["x"].shape
    return out, lam, lam_init


@pytest.mark.parametrize("norm_weights,fused_qkv", [(False, True), (True, True), (False, False)])
def test_layer_small_all_elements(norm_weights, fused_qkv):
    """X [1, 256, 512], h=2, d=128, Dv=256, d_ff=1536: every output element, with and without
    RMSNorm gains (norm2's folded into the W_O epilogue's operand copy) and with one or three
    projection GEMMs."""
    w = gi.WORKLOADS["layer_small_bf16"]
    t = gi.layer_inputs(w, norm_weights=norm_weights)
    out, lam, lam_init = _layer(w, t, fused_qkv=fused_qkv)
    ref = orc.layer_fwd(t["x"], t["w_q"], t["w_k"], t["w_v"], t["w_o"], t["w_gate"], t["w_up"], t["w_down"], w.H,
                        lam, lam_init, w.eps, t.get("norm1_w"), t.get("norm2_w"))
    ma, rr = errors(out, ref)
    print(f"layer small (norm weights {norm_weights}): max-abs {ma:.3e} rel-RMS {rr:.3e}")
    assert_bf16_parity(out, ref, "layer small")
    # The residual branches must both be present: the output is neither X nor X + attention alone.
    assert np.abs(ref - t["x"].double().numpy()).mean() > 0.1


def test_layer_workload_causal_prefix():
    """X [2, 4096, 2048], h=8, d=128, Dv=256, d_ff=5632. The layer is causal, so its
    first 384 output rows depend on the first 384 input rows alone: the oracle computes
    those on the prefix and the full-size GPU output is compared there."""
    w = gi.WORKLOADS["layer_bf16"]
    t = gi.layer_inputs(w)
    out, lam, lam_init = _layer(w, t)
    P = 384
    ref = orc.layer_fwd(t["x"][:, :P], t["w_q"], t["w_k"], t["w_v"], t["w_o"], t["w_gate"], t["w_up"],
                        t["w_down"], w.H, lam, lam_init, w.eps)
    ma, rr = errors(out[:, :P], ref)
    print(f"layer workload prefix: max-abs {ma:.3e} rel-RMS {rr:.3e}")
    assert_bf16_parity(out[:, :P], ref, "layer workload prefix")
    assert torch.isfinite(out).all()


def test_layer_bf16_operands():
    """The layer on the bf16 weights as given, with bf16 GEMM operands. Rounding the
    normalised activations, the attention output and the SwiGLU output to bf16 (half an
    ulp, 2^-9 relative, each) is the whole difference from the fp16-operand run: on the
    small layer it amounts to about 2.1e-3 relative RMS and 1.2e-2 max-abs against the
    float64 layer, so the bound here is 4e-3 relative RMS and 3e-2 max-abs."""
    w = gi.WORKLOADS["layer_small_bf16"]
    t = gi.layer_inputs(w)
    out, lam, lam_init = _layer(w, t, torch.bfloat16)
    ref = orc.layer_fwd(t["x"], t["w_q"], t["w_k"], t["w_v"], t["w_o"], t["w_gate"], t["w_up"], t["w_down"], w.H,
                        lam, lam_init, w.eps)
    ma, rr = errors(out, ref)
    print(f"layer small, bf16 operands: max-abs {ma:.3e} rel-RMS {rr:.3e}")
    assert ma <= 3e-2 and rr <= 4e-3, f"max-abs {ma:.3e}, rel-RMS {rr:.3e}"

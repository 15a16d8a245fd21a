"""GPU parity of diffattn_fwd against the float64 oracle (fp32 CUDA-core path
and bf16 tensor-core path), on seeded inputs."""

import numpy as np
import pytest
import torch

import differential_attention_02_gb300 as da
from differential_attention_02_gb300 import inputs as gi
from oracle import diffattn_oracle as orc
from parity import assert_bf16_out_parity, assert_bf16_parity, assert_f32_parity

pytestmark = pytest.mark.gpu
NAMES = ("q1", "q2", "k1", "k2", "v")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from differential_attention_02_gb300 import build
    build.build()
    da.load_library()


def _lam(w, override=None):
    lv = gi.lambda_vectors(w)
    return orc.reparam_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer, override)


def _run(t, lam, lam_init, eps=1e-5, **kw):
    ws = da.workspace(256)
    out = da.diffattn_fwd(*(t[k].cuda() for k in NAMES), lam, lam_init, eps, ws=ws, **kw)
    assert da.read_error(ws) == 0
    return out


# ------------------------------------------------------------------ fp32 path
def test_tiny_fp32_workload_all_elements():
    w = gi.WORKLOADS["tiny_fp32"]
    t = gi.prefill_inputs(w)
    lam, lam_init = _lam(w)
    ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, lam_init, w.eps)
    assert_f32_parity(_run(t, lam, lam_init, w.eps), ref, "tiny fp32")


@pytest.mark.parametrize("N,d,Dv,causal", [(1, 32, 64, True), (45, 32, 64, True), (70, 64, 128, False),
                                           (33, 128, 256, True), (20, 8, 32, True)])
def test_fp32_shapes(N, d, Dv, causal):
    w = gi.WORKLOADS["tiny_fp32"]
    g = torch.Generator().manual_seed(N * 7 + d)
    t = {k: torch.randn(2, 3, N, Dv if k == "v" else d, generator=g) for k in NAMES}
    lam, lam_init = 0.37, 0.2
    ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, lam_init, 1e-5, causal=causal)
    assert_f32_parity(_run(t, lam, lam_init, causal=causal), ref, f"fp32 N={N} d={d}")


def test_fp32_norm_weight_and_bf16_output():
    w = gi.WORKLOADS["tiny_fp32"]
    t = gi.prefill_inputs(w)
    lam, lam_init = _lam(w)
    nw = torch.linspace(0.5, 1.5, w.Dv)
    ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, lam_init, w.eps, weight=nw.numpy())
    assert_f32_parity(_run(t, lam, lam_init, w.eps, norm_weight=nw.cuda()), ref, "weight")
    out = _run(t, lam, lam_init, w.eps, norm_weight=nw.cuda(), out_dtype=torch.bfloat16)
    d = np.abs(out.float().cpu().numpy() - ref)
    assert np.all(d <= 2.0 ** -8 * np.abs(ref) + 1e-6)  # bf16 rounding of the result only


# ------------------------------------------------------------------ bf16 path
@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 2, 127), (1, 2, 128), (2, 1, 129), (1, 3, 300), (2, 2, 512)])
def test_bf16_prefill_small_and_ragged(B, H, N):
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w, B=B, H=H, N=N)
    lam, lam_init = _lam(w)
    ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, lam_init, w.eps)
    assert_bf16_parity(_run(t, lam, lam_init, w.eps), ref, f"bf16 B{B} H{H} N{N}")


@pytest.mark.parametrize("lam", [0.0, -0.7, 1.0, 2.5])
def test_bf16_lambda_values(lam):
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w, B=1, H=2, N=256)
    ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, 0.5, w.eps)
    assert_bf16_parity(_run(t, lam, 0.5, w.eps), ref, f"lambda {lam}")


def test_bf16_non_causal_weight_and_bf16_out():
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w, B=1, H=2, N=200)
    lam, lam_init = _lam(w)
    nw = torch.linspace(0.5, 1.5, w.Dv)
    ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, lam_init, w.eps, weight=nw.numpy(), causal=False)
    assert_bf16_parity(_run(t, lam, lam_init, w.eps, norm_weight=nw.cuda(), causal=False), ref, "non-causal")
    out = _run(t, lam, lam_init, w.eps, norm_weight=nw.cuda(), causal=False, out_dtype=torch.bfloat16)
    assert_bf16_out_parity(out, ref, "bf16 out")


@pytest.mark.parametrize("d,Dv,in_dtype", [(64, 128, torch.bfloat16), (128, 256, torch.float16)])
def test_f16_output_is_the_rounded_f32_output(d, Dv, in_dtype):
    """The fp16 output path writes exactly the fp32 result rounded to fp16."""
    g = torch.Generator().manual_seed(d + 11)
    t = {k: torch.randn(1, 2, 300, Dv if k == "v" else d, generator=g).to(in_dtype) for k in NAMES}
    out32 = _run(t, 0.45, 0.3)
    out16 = _run(t, 0.45, 0.3, out_dtype=torch.float16)
    assert out16.dtype == torch.float16
    assert torch.equal(out16.cpu(), out32.cpu().half())


@pytest.mark.parametrize("B,H,N,causal,out_dtype", [
    (1, 1, 1, True, torch.bfloat16),      # one query tile, one key tile
    (64, 16, 1, True, torch.float16),     # 1024 query tiles of one key tile each: ~7 per CTA
    (2, 8, 513, True, torch.bfloat16),    # fewer query tiles than SMs, ragged last tile
    (8, 16, 640, True, torch.float16),    # several query tiles per CTA, 1..5 key tiles each
    (4, 16, 1000, False, torch.bfloat16), # non-causal, ragged
    (1, 4, 2944, True, torch.bfloat16),   # largest causal N of the short-sequence (persistent) form
    (1, 4, 3072, True, torch.bfloat16),   # smallest N of the per-tile form
])
def test_16bit_output_forms(B, H, N, causal, out_dtype):
    _check_16bit_output_forms(B, H, N, causal, out_dtype, torch.bfloat16)


@pytest.mark.parametrize("B,H,N,causal", [(4, 16, 300, True), (2, 8, 1000, False)])
def test_16bit_output_forms_fp16_operands(B, H, N, causal):
    """fp16 operands through the persistent kernel (fp16 output) against the per-tile kernel's
    fp32 output, and the oracle."""
    _check_16bit_output_forms(B, H, N, causal, torch.float16, torch.float16)


def _check_16bit_output_forms(B, H, N, causal, out_dtype, in_dtype):
    """16-bit outputs of short sequences come from the persistent kernel (one CTA per SM
    walking query tiles), fp32 outputs from the per-tile kernel; both compute the same fp32
    values, so the 16-bit output is exactly the fp32 output rounded. Small cases also meet
    the oracle."""
    w = gi.WORKLOADS["prefill_bf16"]
    t = {k: v.to(in_dtype) for k, v in gi.prefill_inputs(w, B=B, H=H, N=N).items()}
    lam, lam_init = _lam(w)
    nw = torch.linspace(0.5, 1.5, w.Dv).cuda() if N == 640 else None
    out32 = _run(t, lam, lam_init, w.eps, causal=causal, norm_weight=nw)
    out16 = _run(t, lam, lam_init, w.eps, causal=causal, norm_weight=nw, out_dtype=out_dtype)
    assert torch.equal(out16.cpu(), out32.cpu().to(out_dtype))
    if B * H * N <= 128 * 1024:
        ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, lam_init, w.eps, causal=causal,
                               weight=None if nw is None else nw.cpu().numpy())
        assert_bf16_out_parity(out16, ref, f"{out_dtype} out B{B} H{H} N{N}")


def test_bf16_strided_views():
    """Q1/Q2 and K1/K2 as halves of one [B, N, H, 2d] buffer (the module's layout)."""
    w = gi.WORKLOADS["prefill_bf16"]
    B, H, N, d = 2, 3, 160, 64
    g = torch.Generator().manual_seed(5)
    qk = torch.randn(2, B, N, H, 2 * d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, N, H, 128, generator=g).to(torch.bfloat16)
    q4, k4, v4 = qk[0].permute(0, 2, 1, 3), qk[1].permute(0, 2, 1, 3), v.permute(0, 2, 1, 3)
    t = {"q1": q4[..., :d], "q2": q4[..., d:], "k1": k4[..., :d], "k2": k4[..., d:], "v": v4}
    ref = orc.diffattn_fwd(*(t[k] for k in NAMES), 0.6, 0.3, w.eps)
    dev = {k: x.cuda() for k, x in (("qk", qk), ("v", v))}
    q4d, k4d = dev["qk"][0].permute(0, 2, 1, 3), dev["qk"][1].permute(0, 2, 1, 3)
    out = da.diffattn_fwd(q4d[..., :d], q4d[..., d:], k4d[..., :d], k4d[..., d:], dev["v"].permute(0, 2, 1, 3),
                          0.6, 0.3, w.eps)
    assert_bf16_parity(out, ref, "strided")


def test_bf16_prefill_workload_all_heads():
    """The B=4, H=16, N=2048 prefill workload, every element."""
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w)
    lam, lam_init = _lam(w)
    out = _run(t, lam, lam_init, w.eps)
    ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, lam_init, w.eps)
    assert_bf16_parity(out, ref, "prefill workload")
    outb = _run(t, lam, lam_init, w.eps, out_dtype=torch.bfloat16)
    assert_bf16_out_parity(outb, ref, "prefill workload, bf16 out")


def test_bf16_long_prefill_sampled_rows():
    """The B=1, H=16, N=16384 workload: every head, 40 sampled rows each (incl. first/last)."""
    w = gi.WORKLOADS["long_prefill_bf16"]
    t = gi.prefill_inputs(w)
    lam, lam_init = _lam(w)
    out = _run(t, lam, lam_init, w.eps)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 1], rng.integers(0, w.N, 35)]))
    ref = np.full(out.shape, np.nan)
    for h in range(w.H):
        o = orc.diffattn_head(*(t[k][0, h, rows] if k in ("q1", "q2") else t[k][0, h] for k in NAMES), lam,
                              positions=rows)
        ref[0, rows, h, :] = orc.head_rmsnorm_scale(o, lam_init, w.eps)
    assert_bf16_parity(out, ref, "long prefill")


def test_repeat_calls_are_deterministic():
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w, B=1, H=4, N=640)
    a = _run(t, 0.5, 0.3)
    b = _run(t, 0.5, 0.3)
    assert torch.equal(a, b)


# ------------------------------------------------------------------ wide heads (d=128, Dv=256), CTA-pair kernel
@pytest.mark.parametrize("B,H,N,causal", [(1, 1, 1, True), (1, 2, 129, True), (2, 1, 256, True), (1, 2, 300, False),
                                          (1, 1, 640, True)])
def test_bf16_wide_heads(B, H, N, causal):
    g = torch.Generator().manual_seed(N + 11)
    t = {k: torch.randn(B, H, N, 256 if k == "v" else 128, generator=g).to(torch.bfloat16) for k in NAMES}
    lam, lam_init = 0.63, 0.2
    ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, lam_init, 1e-5, causal=causal)
    assert_bf16_parity(_run(t, lam, lam_init, causal=causal), ref, f"wide B{B} H{H} N{N}")


def test_bf16_wide_heads_weight_bf16_out_and_lambda():
    """The absolute bound is stated for unit gain: with a gain vector it is
    checked on the output divided by the gain (the error scales with it)."""
    g = torch.Generator().manual_seed(77)
    t = {k: torch.randn(1, 3, 200, 256 if k == "v" else 128, generator=g).to(torch.bfloat16) for k in NAMES}
    nw = torch.linspace(0.5, 1.5, 256)
    for lam in (-0.5, 0.0, 1.3):
        ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, 0.4, 1e-5, weight=nw.numpy())
        out = _run(t, lam, 0.4, norm_weight=nw.cuda())
        assert_bf16_parity(out / nw.cuda(), ref / nw.numpy(), f"wide lam {lam}")
        outb = _run(t, lam, 0.4, norm_weight=nw.cuda(), out_dtype=torch.bfloat16)
        assert_bf16_out_parity(outb.float() / nw.cuda(), ref / nw.numpy(), "wide bf16 out")


# ------------------------------------------------------------------ fp16 operands (both kernels)
@pytest.mark.parametrize("d,Dv,N", [(64, 128, 1), (64, 128, 200), (64, 128, 513), (128, 256, 130), (128, 256, 384)])
def test_f16_operands(d, Dv, N):
    g = torch.Generator().manual_seed(d + N)
    t = {k: torch.randn(2, 2, N, Dv if k == "v" else d, generator=g).to(torch.float16) for k in NAMES}
    lam, lam_init = 0.55, 0.3
    ref = orc.diffattn_fwd(*(t[k] for k in NAMES), lam, lam_init, 1e-5)
    assert_bf16_parity(_run(t, lam, lam_init), ref, f"f16 d{d} N{N}")
    assert_bf16_out_parity(_run(t, lam, lam_init, out_dtype=torch.bfloat16), ref, f"f16 d{d} N{N} bf16 out")


def test_host_entry_point_matches_device_call():
    """diffattn_fwd_host (one C-ABI call: pinned host buffers, the batch pipelined over
    copy/compute/copy streams, uneven pieces) returns exactly what one device call returns,
    meets the oracle, and leaves the error word of its staging buffer at zero."""
    w = gi.WORKLOADS["prefill_bf16"]
    host = gi.prefill_inputs(w, B=3, H=2, N=300)
    pin = [host[k].pin_memory() for k in NAMES]
    lam, lam_init = 0.45, 0.47
    for chunks in (None, 1, 2, 3, 6):  # 6: head ranges within each batch entry
        got = da.diffattn_fwd_host(*pin, lam, lam_init, out_dtype=torch.bfloat16, chunks=chunks)
        torch.cuda.synchronize()
        want = da.diffattn_fwd(*(t.cuda() for t in pin), lam, lam_init, out_dtype=torch.bfloat16)
        assert torch.equal(got, want.cpu()), f"chunks={chunks}"
    buf = da.host_buffer_workspace(3, 2, 300, 64, 128, torch.bfloat16, torch.bfloat16, torch.device("cuda", 0))
    assert da.read_error(buf) == 0
    ref = orc.diffattn_fwd(*(host[k] for k in NAMES), lam, lam_init)
    assert_bf16_out_parity(got, ref, "host entry point B3 H2 N300")


def test_host_entry_point_gain_noncausal_fp32_out():
    """The host entry point with a gain (device pointer), the non-causal mask and fp32 output,
    against the device call on the same inputs."""
    w = gi.WORKLOADS["prefill_bf16"]
    host = gi.prefill_inputs(w, B=2, H=3, N=200)
    pin = [host[k].pin_memory() for k in NAMES]
    gain = torch.linspace(0.5, 1.5, 128, device="cuda")
    got = da.diffattn_fwd_host(*pin, 0.6, 0.2, out_dtype=torch.float32, chunks=2, norm_weight=gain, causal=False)
    torch.cuda.synchronize()
    want = da.diffattn_fwd(*(t.cuda() for t in pin), 0.6, 0.2, 1e-5, gain, out_dtype=torch.float32, causal=False)
    assert torch.equal(got, want.cpu())

"""GPU parity of the backward pass (diffattn_bwd) against the float64 oracle's chain
rule of the definition, on seeded inputs.

Two paths, two bars:
- CUDA-core path (fp32 inputs, and every (d, Dv) but (64, 128)): fp32 arithmetic
  from inputs the oracle sees exactly (bf16 and fp16 values are exact in fp32),
  so the bar is fp32 accumulation error: relative RMS <= 2e-5 per gradient tensor
  and max-abs <= 2e-4 of the tensor's largest magnitude; dlambda and dw within
  1e-4 relative.
- Tensor-core path (bf16 or fp16 operands with d = 64, Dv = 128): the products run
  on 16-bit operands, so dO (for dA = dO V^T and dV), A = P1 - lambda P2 (for dV)
  and dS1, dS2 (for dQ, dK) are rounded to the operand type first, as the forward
  rounds P. Each rounding is a relative error of at most half an ulp: 2^-8 for
  bf16 (8 significant bits), 2^-11 for fp16 (11 bits). Measured on the GPU:
  2.3-2.6e-3 relative RMS per gradient tensor for bf16 and 3e-4 for fp16 (max-abs
  up to 4.2e-3 and 4.9e-4 of the tensor's largest value); dw within 1.9e-3
  relative RMS (bf16). The bars are twice the measurement: bf16 5e-3 RMS and 1e-2
  max-abs, fp16 1e-3 and 2e-3; dw 1e-2 (bf16) and 2e-3 (fp16). dlambda has its
  own bar (_dlam_bound): the sum cancels, so its error is bounded against its
  terms, not its value.
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


# (relative RMS, max-abs / max, dlambda and dw relative) per path
BOUNDS = {"fp32": (2e-5, 2e-4, 1e-4), torch.bfloat16: (5e-3, 1e-2, 1e-2), torch.float16: (1e-3, 2e-3, 2e-3)}


def _bounds(d, Dv, dtype):
    """The tensor-core path serves bf16/fp16 operands with d = 64, Dv = 128."""
    return BOUNDS[dtype] if (d, Dv) == (64, 128) and dtype in (torch.bfloat16, torch.float16) else BOUNDS["fp32"]


def _check(g, ref, what, heads=None, bounds=BOUNDS["fp32"]):
    rr_max, ma_max, _ = bounds
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
        assert rr <= rr_max and ma <= ma_max, f"{what} {k}: rel-RMS {rr:.3e}, max-abs/max {ma:.3e}"


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
    (1, 2, 300, 64, 128, True, torch.float16),
    (1, 1, 1, 64, 128, True, torch.bfloat16),
    (1, 2, 512, 64, 128, False, torch.float16),
])
def test_backward_shapes(B, H, N, d, Dv, causal, dtype):
    g0 = torch.Generator().manual_seed(B * 1000 + N * 7 + d)
    t = {k: torch.randn(B, H, N, Dv if k == "v" else d, generator=g0).to(dtype) for k in NAMES}
    dy = torch.randn(B, N, H, Dv, generator=g0).to(dtype)
    lam, lam_init = 0.58, 0.35
    g = _run(t, dy, lam, lam_init, causal=causal, want_dnorm_weight=True)
    ref = orc.diffattn_bwd(*(t[k] for k in NAMES), dy, lam, lam_init, 1e-5, causal=causal)
    bounds = _bounds(d, Dv, dtype)
    _check(g, ref, f"B{B} H{H} N{N} d{d} {dtype}", bounds=bounds)
    _check_sums(g, ref, bounds, t, dy, lam, lam_init, causal=causal)


def _dlam_bound(t, dy, lam, lam_init, u, eps=1e-5, weight=None, causal=True):
    """Error bar for dlambda = -sum_ij dA_ij P2_ij on the tensor-core path.

    The sum cancels almost completely (a row's dO is orthogonal to its normalised output),
    so its error is set by the terms t_ij = dA_ij P2_ij, not by the result. P2 reaches the
    sum through P2 V, which the forward forms from P rounded to the operand type: term
    t_ij carries a relative error of at most u (2^-8 bf16, 2^-11 fp16), of standard
    deviation at most u / sqrt(3), independently from term to term; the bar is four
    standard deviations of that sum, sqrt(sum t_ij^2) u 4 / sqrt(3), plus 2^-20 of
    sum |dO_ic| P2_ij |V_jc| for the fp32 arithmetic of dO and the sums. Measured errors
    are 0.3-0.6 of one standard deviation; a flipped sign of dlambda exceeds the bar on
    every case here. dO, dA and P2 come from the oracle's primitives in float64."""
    B, H, N, d = t["q1"].shape
    sq, mag = 0.0, 0.0
    for b in range(B):
        for h in range(H):
            q1, q2, k1, k2, v = (t[k][b, h] for k in NAMES)
            o = orc.diffattn_head(q1, q2, k1, k2, v, lam, causal)
            allowed = orc.causal_allowed(np.arange(N), N) if causal else np.ones((N, N), bool)
            q2d, k2d, vd = (x.double().numpy() for x in (q2, k2, v))
            p2 = orc.masked_softmax_rows((q2d @ k2d.T) / np.sqrt(d), allowed)
            r = np.sqrt(np.mean(o * o, axis=1, keepdims=True) + eps)
            n = o / r
            gg = dy[b, :, h, :].double().numpy() * (1.0 if weight is None else weight) * (1.0 - lam_init)
            d_o = (gg - n * np.mean(gg * n, axis=1, keepdims=True)) / r
            terms = (d_o @ vd.T) * p2
            sq += float(np.sum(terms * terms))
            mag += float(np.sum((np.abs(d_o) @ np.abs(vd).T) * p2))
    return 4.0 * u / np.sqrt(3.0) * np.sqrt(sq) + 2.0 ** -20 * mag


def _check_sums(g, ref, bounds, t=None, dy=None, lam=None, lam_init=None, **kw):
    rel = bounds[2]
    got = float(g["dlam"].item())
    dw, dw_ref = g["dw"].cpu().double().numpy(), ref["dw"]
    if rel > 1e-4:  # tensor-core path
        u = 2.0 ** -8 if rel >= 1e-2 else 2.0 ** -11
        bar = _dlam_bound(t, dy, lam, lam_init, u, **kw)
        print(f"dlambda {got:.6g} vs {ref['dlam']:.6g}: |err| {abs(got - ref['dlam']):.3e}, bar {bar:.3e}")
        assert abs(got - ref["dlam"]) <= bar
        assert np.linalg.norm(dw - dw_ref) <= rel * np.linalg.norm(dw_ref)  # relative RMS of the vector
    else:
        assert got == pytest.approx(ref["dlam"], rel=rel, abs=1e-6)
        np.testing.assert_allclose(dw, dw_ref, rtol=rel, atol=1e-5)


@pytest.mark.parametrize("lam", [0.0, -0.8, 2.2])
def test_backward_lambda_values_and_norm_weight(lam):
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w, B=1, H=2, N=200)
    dy = gi.output_grad(w, B=1, H=2, N=200)
    nw = torch.linspace(0.5, 1.5, w.Dv)
    g = _run(t, dy, lam, 0.4, norm_weight=nw.cuda(), want_dnorm_weight=True)
    ref = orc.diffattn_bwd(*(t[k] for k in NAMES), dy, lam, 0.4, 1e-5, weight=nw.numpy())
    bounds = _bounds(w.d, w.Dv, t["q1"].dtype)
    _check(g, ref, f"lambda {lam}", bounds=bounds)
    _check_sums(g, ref, bounds, t, dy, lam, 0.4, weight=nw.numpy())
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
    _check(g, ref, "strided", bounds=_bounds(d, 128, torch.bfloat16))


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
    bounds = _bounds(w.d, w.Dv, t["q1"].dtype)
    _check(g, ref, "prefill workload", heads=heads, bounds=bounds)
    _check_sums(g, ref, bounds, t, dy, lam, lam_init, eps=w.eps)


@pytest.mark.parametrize("B,H,N,causal,dtype,weight", [
    (1, 1, 1, True, torch.bfloat16, False),
    (1, 3, 130, True, torch.bfloat16, True),
    (2, 2, 300, False, torch.float16, False),
    (1, 2, 513, True, torch.float16, True),
])
def test_training_pair(B, H, N, causal, dtype, weight):
    """diffattn_fwd_train returns diffattn_fwd's output bit for bit. The backward from its saved
    state meets the oracle with the tensor-core path's bars and agrees with the recomputing
    backward to 1e-3 relative RMS per gradient (bf16; 2e-4 fp16) plus one rounding to the
    operand type (u / sqrt(3) relative RMS, u = 2^-8 bf16, 2^-11 fp16): the same operands and
    products, except that the saved O2/l2 carries that one rounding (it enters D1 and D2
    linearly, not the norm), and the fp32 order of the per-row sums differs (and with it,
    rarely, which way an element of dO rounds to the operand type)."""
    g0 = torch.Generator().manual_seed(B * 100 + N)
    t = {k: torch.randn(B, H, N, 128 if k == "v" else 64, generator=g0).to(dtype) for k in NAMES}
    dy = torch.randn(B, N, H, 128, generator=g0).to(dtype)
    dev = {k: v.cuda() for k, v in t.items()}
    nw = torch.linspace(0.5, 1.5, 128) if weight else None
    nwd = None if nw is None else nw.cuda()
    lam, lam_init = 0.58, 0.35
    saved = None
    for out_dtype in (torch.float32, dtype):
        ref = da.diffattn_fwd(*(dev[k] for k in NAMES), lam, lam_init, norm_weight=nwd, causal=causal,
                              out_dtype=out_dtype)
        out, saved = da.diffattn_fwd_train(*(dev[k] for k in NAMES), lam, lam_init, norm_weight=nwd, causal=causal,
                                           out_dtype=out_dtype, saved=saved)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"training forward output, {out_dtype}"
    kw = dict(norm_weight=nwd, causal=causal, want_dnorm_weight=True)
    a = da.diffattn_bwd(*(dev[k] for k in NAMES), dy.cuda(), lam, lam_init, **kw)
    a = {k: v.clone() for k, v in a.items()}
    ws = da.workspace(da.bwd_workspace_bytes(B, H, N, 64, 128))
    g = da.diffattn_bwd(*(dev[k] for k in NAMES), dy.cuda(), lam, lam_init, saved=saved, ws=ws, **kw)
    torch.cuda.synchronize()
    assert da.read_error(ws) == 0
    ref = orc.diffattn_bwd(*(t[k] for k in NAMES), dy, lam, lam_init, 1e-5, causal=causal,
                           weight=None if nw is None else nw.numpy())
    bounds = _bounds(64, 128, dtype)
    _check(g, ref, f"from saved state B{B} H{H} N{N}", bounds=bounds)
    _check_sums(g, ref, bounds, t, dy, lam, lam_init, causal=causal, weight=None if nw is None else nw.numpy())
    tol = 1e-3 + 2.0 ** -8 / np.sqrt(3) if dtype == torch.bfloat16 else 2e-4 + 2.0 ** -11 / np.sqrt(3)
    for k in GRADS + ("dw",):
        x, y = g[k].double(), a[k].double()
        rr = float((x - y).norm() / y.norm().clamp_min(1e-30))
        print(f"{k}: saved vs recompute rel-RMS {rr:.2e}")
        assert rr <= tol or float((x - y).abs().max()) <= 1e-6, f"{k}: saved vs recompute rel-RMS {rr:.2e}"


@pytest.mark.parametrize("lam,dtype", [(0.0, torch.bfloat16), (-0.7, torch.float16), (2.2, torch.bfloat16)])
def test_training_pair_lambda_values(lam, dtype):
    """The saved state's O1/l1 is rebuilt as x + lambda O2/l2, so lambda enters the backward's
    preparation directly: the training pair against the oracle at lambda = 0 (O2/l2 drops out;
    dQ2 and dK2 are exactly zero), lambda < 0 and lambda > 1, with a gain."""
    B, H, N = 1, 2, 200
    g0 = torch.Generator().manual_seed(int(1000 * abs(lam)) + 7)
    t = {k: torch.randn(B, H, N, 128 if k == "v" else 64, generator=g0).to(dtype) for k in NAMES}
    dy = torch.randn(B, N, H, 128, generator=g0).to(dtype)
    nw = torch.linspace(0.5, 1.5, 128)
    dev = {k: v.cuda() for k, v in t.items()}
    lam_init = 0.35
    _, saved = da.diffattn_fwd_train(*(dev[k] for k in NAMES), lam, lam_init, norm_weight=nw.cuda())
    ws = da.workspace(da.bwd_workspace_bytes(B, H, N, 64, 128))
    g = da.diffattn_bwd(*(dev[k] for k in NAMES), dy.cuda(), lam, lam_init, norm_weight=nw.cuda(),
                        want_dnorm_weight=True, ws=ws, saved=saved)
    torch.cuda.synchronize()
    assert da.read_error(ws) == 0
    ref = orc.diffattn_bwd(*(t[k] for k in NAMES), dy, lam, lam_init, 1e-5, weight=nw.numpy())
    bounds = _bounds(64, 128, dtype)
    _check(g, ref, f"training pair lambda {lam}", bounds=bounds)
    _check_sums(g, ref, bounds, t, dy, lam, lam_init, weight=nw.numpy())
    if lam == 0.0:
        assert float(g["dq2"].abs().max()) == 0.0 and float(g["dk2"].abs().max()) == 0.0


def test_training_forward_saved_state_against_the_definition():
    """The saved state pinned to the definition, independently of the backward: with
    A_m = softmax_m V (each map's attention output, float64), x = A1 - lambda A2 (fp32),
    A2 in the operand type, and L_m = log2 sum_j exp2(S_ij log2(e) / sqrt(d)) (the row's
    log-sum-exp in base 2 of the scaled scores). P enters the PV products rounded to the
    operand type (the forward's 3e-3 relative RMS bar); A2 is rounded once more (at most
    u = 2^-8 bf16 or 2^-11 fp16 relative, u / sqrt(3) RMS); L only sees fp32 sums, exp2 and
    log2: 1e-4 absolute."""
    for in_dtype in (torch.bfloat16, torch.float16):
        w = gi.WORKLOADS["prefill_bf16"]
        B, H, N = 1, 2, 300
        lam = 0.5
        t = gi.prefill_inputs(w, B=B, H=H, N=N)
        ops = [t[k].to(in_dtype).cuda() for k in NAMES]
        _, saved = da.diffattn_fwd_train(*ops, lam, 0.3, w.eps)
        torch.cuda.synchronize()
        rows = B * H * N
        r256 = lambda n: (n + 255) // 256 * 256
        xb, ab = rows * w.Dv * 4, rows * w.Dv * 2
        x = saved[:xb].view(torch.float32).view(B, H, N, w.Dv).double().cpu().numpy()
        a2 = saved[r256(xb):r256(xb) + ab].view(in_dtype).view(B, H, N, w.Dv).double().cpu().numpy()
        off = r256(xb) + r256(ab)
        lse = saved[off:off + rows * 8].view(torch.float32).view(B, H, N, 2).double().cpu().numpy()
        allowed = orc.causal_allowed(np.arange(N), N)
        u = 2.0 ** -8 if in_dtype == torch.bfloat16 else 2.0 ** -11
        rel = lambda got, ref: np.linalg.norm(got - ref) / np.linalg.norm(ref)
        for h in range(H):
            v = ops[4][0, h].double().cpu().numpy()
            ref_a, ref_l = [], []
            for qi, ki in ((0, 2), (1, 3)):
                s = ops[qi][0, h].double().cpu().numpy() @ ops[ki][0, h].double().cpu().numpy().T / np.sqrt(w.d)
                ref_a.append(orc.masked_softmax_rows(s, allowed) @ v)
                z = np.where(allowed, s, -np.inf) * np.log2(np.e)
                mx = z.max(axis=1)
                ref_l.append(mx + np.log2(np.exp2(z - mx[:, None]).sum(axis=1)))
            rx = rel(x[0, h], ref_a[0] - lam * ref_a[1])
            ra = rel(a2[0, h], ref_a[1])
            assert rx <= 3e-3, f"{in_dtype} head {h}: x rel-RMS {rx:.2e}"
            assert ra <= 3e-3 + u / np.sqrt(3), f"{in_dtype} head {h}: O2/l2 rel-RMS {ra:.2e}"
            for m in range(2):
                assert np.abs(lse[0, h, :, m] - ref_l[m]).max() <= 1e-4, f"{in_dtype} head {h} map {m + 1}: L"


def test_training_forward_saved_state_prefill_workload_sampled_heads():
    """The saved state at the full B=4, H=16, N=2048 prefill workload, on three heads against
    the definition (x, O2/l2 and L as in the test above, the same bars), and its size."""
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w)
    lam = 0.5
    dev = {k: v.cuda() for k, v in t.items()}
    _, saved = da.diffattn_fwd_train(*(dev[k] for k in NAMES), lam, 0.3, w.eps, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    rows = w.B * w.H * w.N
    r256 = lambda n: (n + 255) // 256 * 256
    xb, ab = rows * w.Dv * 4, rows * w.Dv * 2
    assert saved.numel() == r256(xb) + r256(ab) + r256(rows * 8)
    allowed = orc.causal_allowed(np.arange(w.N), w.N)
    for b, h in ((0, 0), (1, 7), (3, 15)):
        row0 = (b * w.H + h) * w.N
        x = saved[row0 * w.Dv * 4:(row0 + w.N) * w.Dv * 4].view(torch.float32).view(w.N, w.Dv).double().cpu().numpy()
        a2 = saved[r256(xb) + row0 * w.Dv * 2:r256(xb) + (row0 + w.N) * w.Dv * 2].view(torch.bfloat16)
        a2 = a2.view(w.N, w.Dv).double().cpu().numpy()
        off = r256(xb) + r256(ab)
        lse = saved[off + row0 * 8:off + (row0 + w.N) * 8].view(torch.float32).view(w.N, 2).double().cpu().numpy()
        v = t["v"][b, h].double().numpy()
        ref_a, ref_l = [], []
        for qn, kn in (("q1", "k1"), ("q2", "k2")):
            sc = t[qn][b, h].double().numpy() @ t[kn][b, h].double().numpy().T / np.sqrt(w.d)
            ref_a.append(orc.masked_softmax_rows(sc, allowed) @ v)
            z = np.where(allowed, sc, -np.inf) * np.log2(np.e)
            mx = z.max(axis=1)
            ref_l.append(mx + np.log2(np.exp2(z - mx[:, None]).sum(axis=1)))
        rel = lambda got, ref: np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel(x, ref_a[0] - lam * ref_a[1]) <= 3e-3, (b, h)
        assert rel(a2, ref_a[1]) <= 3e-3 + 2.0 ** -8 / np.sqrt(3), (b, h)
        for m in range(2):
            assert np.abs(lse[:, m] - ref_l[m]).max() <= 1e-4, (b, h, m)


def test_training_pair_prefill_workload_sampled_heads():
    """The B=4, H=16, N=2048 prefill workload through the training pair: every gradient of
    three heads against the oracle, and dlambda, dw over all 64 heads."""
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w)
    dy = gi.output_grad(w)
    lv = gi.lambda_vectors(w)
    lam, lam_init = orc.reparam_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer)
    dev = {k: v.cuda() for k, v in t.items()}
    _, saved = da.diffattn_fwd_train(*(dev[k] for k in NAMES), lam, lam_init, w.eps, out_dtype=torch.bfloat16)
    ws = da.workspace(da.bwd_workspace_bytes(w.B, w.H, w.N, w.d, w.Dv))
    g = da.diffattn_bwd(*(dev[k] for k in NAMES), dy.cuda(), lam, lam_init, w.eps, want_dnorm_weight=True, ws=ws,
                        saved=saved)
    torch.cuda.synchronize()
    assert da.read_error(ws) == 0
    heads = [(0, 0), (1, 7), (3, 15)]
    ref = orc.diffattn_bwd(*(t[k] for k in NAMES), dy, lam, lam_init, w.eps)
    bounds = _bounds(w.d, w.Dv, t["q1"].dtype)
    _check(g, ref, "prefill workload from the saved state", heads=heads, bounds=bounds)
    _check_sums(g, ref, bounds, t, dy, lam, lam_init, eps=w.eps)

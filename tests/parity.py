"""Tolerances and comparison helpers for GPU-vs-oracle parity tests.

bf16 inputs with fp32 accumulation: max-abs <= 1e-2 and relative RMS
(||gpu - ref||_2 / ||ref||_2) <= 3e-3. fp32 inputs: max-abs <= 1e-5.
bf16 OUTPUTS: the rounding of the result itself is up to half a bf16 ulp
(<= 2^-8 |ref|), which alone exceeds 1e-2 for |ref| above about 2.5, so the
max-abs bound is applied to |gpu - ref| - 2^-8 |ref|; rel-RMS stays 3e-3.
"""

import numpy as np

BF16_MAX_ABS = 1e-2
BF16_REL_RMS = 3e-3
F32_MAX_ABS = 1e-5


def errors(gpu, ref):
    g = gpu.detach().cpu().double().numpy() if hasattr(gpu, "detach") else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    mask = ~np.isnan(r)  # NaN marks entries the oracle did not compute (sampled checks)
    assert mask.any()
    d = g[mask] - r[mask]
    assert np.all(np.isfinite(g[mask])), "non-finite GPU output"
    return float(np.max(np.abs(d))), float(np.linalg.norm(d) / max(np.linalg.norm(r[mask]), 1e-300))


def assert_bf16_parity(gpu, ref, what=""):
    ma, rr = errors(gpu, ref)
    assert ma <= BF16_MAX_ABS and rr <= BF16_REL_RMS, f"{what}: max-abs {ma:.3e}, rel-RMS {rr:.3e}"
    return ma, rr


def assert_f32_parity(gpu, ref, what=""):
    ma, rr = errors(gpu, ref)
    assert ma <= F32_MAX_ABS, f"{what}: max-abs {ma:.3e}, rel-RMS {rr:.3e}"
    return ma, rr


def assert_bf16_out_parity(gpu, ref, what=""):
    g = gpu.detach().cpu().double().numpy()
    r = np.asarray(ref, np.float64)
    mask = ~np.isnan(r)
    excess = float(np.max(np.abs(g[mask] - r[mask]) - 2.0 ** -8 * np.abs(r[mask])))
    _, rr = errors(gpu, ref)
    assert excess <= BF16_MAX_ABS and rr <= BF16_REL_RMS, f"{what}: max-abs beyond half-ulp {excess:.3e}, rel-RMS {rr:.3e}"
    return excess, rr

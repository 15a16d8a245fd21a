"""Pins for the float64 oracle against facts fixed outside it.

Each test checks the oracle against something other than itself: values the
pages state, closed forms, a library routine (torch's float64 scaled dot-product
attention), definitional invariants, or brute-force loops on tiny inputs. The
set is chosen so that a dropped term, a wrong sign, a wrong scale, a swapped
operand pair or a wrong mask fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import diffattn_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _sdpa_causal(q, k, v):
    """Library routine: torch's float64 CPU causal scaled dot-product attention."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True)[0, 0].numpy()


# ----------------------------------------------------------------- lambda ---

def test_lambda_init_matches_page_values():
    g = json.load(open(os.path.join(GOLDEN, "lambda_init_pages.json")))
    assert orc.lambda_init_schedule(1) == pytest.approx(g["lambda_init_first_layer"], abs=1e-15)
    assert orc.lambda_init_schedule(400) == pytest.approx(g["lambda_init_deep_limit"], abs=1e-15)
    vals = [orc.lambda_init_schedule(l) for l in range(1, 40)]
    assert all(b > a for a, b in zip(vals, vals[1:])), "lower in early layers, higher in deep ones"
    assert all(v < g["lambda_init_deep_limit"] for v in vals)
    lam, lam_init = orc.reparam_lambda(np.zeros(8), np.zeros(8), np.zeros(8), np.zeros(8), layer=5,
                                       lambda_init_override=g["lambda_init_constant_ablation"])
    assert lam_init == 0.8 and lam == pytest.approx(0.8, abs=1e-15)
    with pytest.raises(ValueError):
        orc.lambda_init_schedule(0)


def test_lambda_reparam_closed_forms():
    z = np.zeros(16)
    for l in (1, 3, 6, 12, 24):
        lam, lam_init = orc.reparam_lambda(z, z, z, z, layer=l)
        assert lam == pytest.approx(lam_init, abs=1e-15), "exp(0) - exp(0) cancels"
    # lq1.lk1 = ln 3 and lq2.lk2 = ln 2 give 3 - 2 + lambda_init: fixes both exponentials' signs.
    e0 = np.zeros(4)
    e0[0] = 1.0
    lam, lam_init = orc.reparam_lambda(e0 * math.log(3.0), e0, e0 * 0.5, e0 * 2 * math.log(2.0), layer=1)
    assert lam_init == pytest.approx(0.2, abs=1e-15)
    assert lam == pytest.approx(1.2, abs=1e-13)
    # The dot product runs over the whole vectors: spread ln 3 over 4 entries.
    lam, _ = orc.reparam_lambda(np.full(4, 0.5), np.full(4, math.log(3.0) / 2), z[:4], z[:4], layer=1)
    assert lam == pytest.approx(3.0 - 1.0 + 0.2, abs=1e-13)


# ------------------------------------------------------- mask and softmax ---

def test_masked_softmax_rows_sum_to_one_and_mask_future():
    rng = _rng(0)
    n = 37
    s = rng.normal(size=(n, n)) * 3
    p = orc.masked_softmax_rows(s, orc.causal_allowed(np.arange(n), n))
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(p[np.triu_indices(n, 1)] == 0.0)
    assert np.all(p[np.tril_indices(n)] > 0.0)
    assert p[0, 0] == 1.0


def test_two_token_closed_form_fixes_sqrt_d_scale():
    # d = 4, q = 1s, k0 = 0, k1 = (ln 3 / 2) * 1s: q.k1 / sqrt(4) = ln 3, so row 1 weights are (1/4, 3/4).
    d = 4
    q = np.ones((2, d))
    k = np.zeros((2, d))
    k[1] = math.log(3.0) / 2
    v = np.array([[1.0, 0.0, 2.0], [0.0, 1.0, -2.0]])
    o = orc.diffattn_head(q, q, k, k, v, lam=0.0)
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    np.testing.assert_allclose(o[1], 0.25 * v[0] + 0.75 * v[1], atol=1e-14)


# --------------------------------------------- structure against library ---

@pytest.mark.parametrize("n,d,dv,lam", [(1, 8, 16, 0.3), (33, 16, 32, 0.0), (70, 32, 64, 0.7), (130, 8, 16, -0.4)])
def test_head_is_difference_of_two_library_attentions(n, d, dv, lam):
    """(P1 - lam P2) V = SDPA(q1,k1,v) - lam SDPA(q2,k2,v): pins pairing, scale, mask and sign."""
    rng = _rng(n)
    q1, q2, k1, k2 = (rng.normal(size=(n, d)) for _ in range(4))
    v = rng.normal(size=(n, dv))
    got = orc.diffattn_head(q1, q2, k1, k2, v, lam)
    want = _sdpa_causal(q1, k1, v) - lam * _sdpa_causal(q2, k2, v)
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=1e-12)


def test_lambda_zero_is_standard_causal_attention():
    rng = _rng(5)
    q1, q2, k1, k2 = (rng.normal(size=(50, 16)) for _ in range(4))
    v = rng.normal(size=(50, 24))
    got = orc.diffattn_head(q1, q2, k1, k2, v, 0.0)
    np.testing.assert_allclose(got, _sdpa_causal(q1, k1, v), atol=1e-13)
    # the second map has no influence at lambda = 0
    got2 = orc.diffattn_head(q1, rng.normal(size=(50, 16)), k1, rng.normal(size=(50, 16)), v, 0.0)
    np.testing.assert_array_equal(got, got2)


def test_identical_maps_scale_standard_attention_by_one_minus_lambda():
    rng = _rng(6)
    q, k = rng.normal(size=(40, 8)), rng.normal(size=(40, 8))
    v = rng.normal(size=(40, 12))
    for lam in (0.2, 0.8, 1.0, 1.7):
        got = orc.diffattn_head(q, q, k, k, v, lam)
        np.testing.assert_allclose(got, (1 - lam) * _sdpa_causal(q, k, v), atol=1e-13)


def test_non_causal_option_matches_library():
    rng = _rng(7)
    q1, q2, k1, k2 = (rng.normal(size=(20, 8)) for _ in range(4))
    v = rng.normal(size=(20, 8))
    t = lambda a: torch.from_numpy(a)[None, None]
    sd = lambda q, k: torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v))[0, 0].numpy()
    got = orc.diffattn_head(q1, q2, k1, k2, v, 0.5, causal=False)
    np.testing.assert_allclose(got, sd(q1, k1) - 0.5 * sd(q2, k2), atol=1e-13)


def test_row_chunking_is_exact():
    rng = _rng(8)
    q1, q2, k1, k2 = (rng.normal(size=(90, 8)) for _ in range(4))
    v = rng.normal(size=(90, 8))
    a = orc.diffattn_head(q1, q2, k1, k2, v, 0.6, row_chunk=512)
    b = orc.diffattn_head(q1, q2, k1, k2, v, 0.6, row_chunk=7)
    np.testing.assert_allclose(a, b, atol=1e-14)


def test_row_positions_select_exact_rows():
    rng = _rng(18)
    q1, q2, k1, k2 = (rng.normal(size=(60, 8)) for _ in range(4))
    v = rng.normal(size=(60, 8))
    full = orc.diffattn_head(q1, q2, k1, k2, v, 0.4)
    rows = np.array([0, 7, 31, 59])
    part = orc.diffattn_head(q1[rows], q2[rows], k1, k2, v, 0.4, positions=rows)
    np.testing.assert_array_equal(part, full[rows])


# ------------------------------------------------------ norm and scale ---

def test_rmsnorm_row_rms_and_weight():
    rng = _rng(9)
    o = rng.normal(size=(25, 64)) * rng.uniform(0.01, 5, size=(25, 1))
    eps = 1e-5
    for lam_init in (0.2, 0.666, 0.8):
        y = orc.head_rmsnorm_scale(o, lam_init, eps)
        ms = np.mean(o * o, axis=1)
        np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)),
                                   abs(1 - lam_init) * np.sqrt(ms / (ms + eps)), rtol=1e-12)
        # direction of each row is preserved
        cos = np.sum(y * o, axis=1) / np.linalg.norm(y, axis=1) / np.linalg.norm(o, axis=1)
        np.testing.assert_allclose(cos, 1.0, atol=1e-12)
    w = rng.uniform(0.5, 2.0, size=64)
    np.testing.assert_allclose(orc.head_rmsnorm_scale(o, 0.3, eps, w), orc.head_rmsnorm_scale(o, 0.3, eps) * w,
                               rtol=1e-13)
    assert np.all(orc.head_rmsnorm_scale(np.zeros((2, 8)), 0.3, eps) == 0.0)


def test_first_row_closed_form():
    """Token 0 sees only itself, so O_hat_0 = (1 - lam) V_0 and y_0 has a closed form."""
    rng = _rng(10)
    B, H, N, d, Dv = 2, 3, 9, 8, 16
    q1, q2, k1, k2 = (rng.normal(size=(B, H, N, d)) for _ in range(4))
    v = rng.normal(size=(B, H, N, Dv))
    lam, lam_init, eps = 0.45, 0.3, 1e-5
    out = orc.diffattn_fwd(q1, q2, k1, k2, v, lam, lam_init, eps)
    o0 = (1 - lam) * v[:, :, 0, :]
    y0 = o0 / np.sqrt(np.mean(o0 ** 2, axis=-1, keepdims=True) + eps) * (1 - lam_init)
    np.testing.assert_allclose(out[:, 0, :, :], y0, atol=1e-13)


def test_identical_maps_with_lambda_one_give_zero_output():
    rng = _rng(11)
    q, k = rng.normal(size=(1, 1, 12, 8)), rng.normal(size=(1, 1, 12, 8))
    v = rng.normal(size=(1, 1, 12, 8))
    out = orc.diffattn_fwd(q, q, k, k, v, 1.0, 0.5)
    assert np.max(np.abs(out)) < 1e-10


# --------------------------------------------------- causality, layout ---

def test_causality_later_tokens_do_not_change_earlier_rows():
    rng = _rng(12)
    B, H, N, d, Dv = 1, 2, 40, 8, 8
    t = [rng.normal(size=(B, H, N, d)) for _ in range(4)] + [rng.normal(size=(B, H, N, Dv))]
    base = orc.diffattn_fwd(*t, 0.6, 0.4)
    cut = 23
    t2 = [a.copy() for a in t]
    for a in t2:
        a[:, :, cut:] = rng.normal(size=a[:, :, cut:].shape) * 10
    pert = orc.diffattn_fwd(*t2, 0.6, 0.4)
    np.testing.assert_array_equal(base[:, :cut], pert[:, :cut])
    assert np.max(np.abs(base[:, cut:] - pert[:, cut:])) > 1e-3


def test_output_layout_is_tokens_then_heads():
    rng = _rng(13)
    B, H, N, d, Dv = 2, 3, 5, 4, 6
    t = [rng.normal(size=(B, H, N, d)) for _ in range(4)] + [rng.normal(size=(B, H, N, Dv))]
    out = orc.diffattn_fwd(*t, 0.3, 0.2)
    assert out.shape == (B, N, H, Dv)
    b, h = 1, 2
    one = orc.head_rmsnorm_scale(orc.diffattn_head(*(a[b, h] for a in t), 0.3), 0.2)
    np.testing.assert_array_equal(out[b, :, h, :], one)


# ---------------------------------------------------------- brute force ---

def _brute_force_fwd(q1, q2, k1, k2, v, lam, lam_init, eps):
    """Scalar loops with math.exp: the definition entry by entry."""
    B, H, N, d = q1.shape
    Dv = v.shape[-1]
    out = np.zeros((B, N, H, Dv))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                w = []
                for q, k in ((q1, k1), (q2, k2)):
                    s = [sum(q[b, h, i, c] * k[b, h, j, c] for c in range(d)) / math.sqrt(d) for j in range(i + 1)]
                    mx = max(s)
                    e = [math.exp(x - mx) for x in s]
                    tot = sum(e)
                    w.append([x / tot for x in e])
                o = [sum((w[0][j] - lam * w[1][j]) * v[b, h, j, c] for j in range(i + 1)) for c in range(Dv)]
                rms = math.sqrt(sum(x * x for x in o) / Dv + eps)
                for c in range(Dv):
                    out[b, i, h, c] = o[c] / rms * (1 - lam_init)
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_brute_force_tiny(seed):
    rng = _rng(100 + seed)
    B, H, N, d, Dv = 1, 2, 11, 3, 5
    t = [rng.normal(size=(B, H, N, d)) for _ in range(4)] + [rng.normal(size=(B, H, N, Dv))]
    lam, lam_init = orc.reparam_lambda(*(rng.normal(size=3) * 0.3 for _ in range(4)), layer=3)
    got = orc.diffattn_fwd(*t, lam, lam_init, 1e-5)
    np.testing.assert_allclose(got, _brute_force_fwd(*t, lam, lam_init, 1e-5), atol=1e-12)


# --------------------------------------------------------------- decode ---

def test_decode_equals_last_prefill_row_and_respects_seq_lens():
    rng = _rng(14)
    B, H, L, d, Dv = 3, 2, 30, 8, 16
    k1, k2 = rng.normal(size=(B, H, L, d)), rng.normal(size=(B, H, L, d))
    v = rng.normal(size=(B, H, L, Dv))
    q1, q2 = rng.normal(size=(B, H, L, d)), rng.normal(size=(B, H, L, d))
    lens = [30, 1, 17]
    k1n, k2n, vn = k1.copy(), k2.copy(), v.copy()
    for b, Lb in enumerate(lens):  # entries past each length must be ignored
        k1n[b, :, Lb:] = np.nan
        k2n[b, :, Lb:] = np.nan
        vn[b, :, Lb:] = np.nan
    qd1 = np.stack([q1[b, :, lens[b] - 1] for b in range(B)])
    qd2 = np.stack([q2[b, :, lens[b] - 1] for b in range(B)])
    got = orc.diffattn_decode(qd1, qd2, k1n, k2n, vn, lens, 0.55, 0.47)
    assert np.all(np.isfinite(got))
    for b, Lb in enumerate(lens):
        pre = orc.diffattn_fwd(q1[b:b + 1, :, :Lb], q2[b:b + 1, :, :Lb], k1[b:b + 1, :, :Lb],
                               k2[b:b + 1, :, :Lb], v[b:b + 1, :, :Lb], 0.55, 0.47)
        np.testing.assert_allclose(got[b], pre[0, Lb - 1], atol=1e-12)


# --------------------------------------------------------------- module ---

def test_module_with_identity_projections_reduces_to_heads():
    rng = _rng(15)
    B, N, h, d = 1, 10, 2, 4
    dm = 2 * d * h
    Dv = dm // h
    x = rng.normal(size=(B, N, dm))
    eye = np.eye(dm)
    y = orc.module_fwd(x, eye, eye, eye, eye, h, 0.4, 0.3)
    for i in range(h):
        xs = x[0, :, 2 * d * i: 2 * d * (i + 1)]
        o = orc.diffattn_head(xs[:, :d], xs[:, d:], xs[:, :d], xs[:, d:], x[0, :, Dv * i: Dv * (i + 1)], 0.4)
        np.testing.assert_allclose(y[0, :, Dv * i: Dv * (i + 1)], orc.head_rmsnorm_scale(o, 0.3), atol=1e-13)


def test_module_projection_orientation_and_output_linearity():
    rng = _rng(16)
    B, N, h, d, Dv, dm = 2, 7, 2, 4, 8, 12
    x = rng.normal(size=(B, N, dm))
    wq, wk = rng.normal(size=(dm, 2 * d * h)), rng.normal(size=(dm, 2 * d * h))
    wv, wo = rng.normal(size=(dm, Dv * h)), rng.normal(size=(Dv * h, dm))
    y = orc.module_fwd(x, wq, wk, wv, wo, h, 0.5, 0.2)
    y_cat = orc.module_fwd(x, wq, wk, wv, np.eye(Dv * h), h, 0.5, 0.2)
    np.testing.assert_allclose(y, y_cat @ wo, atol=1e-12)
    # Projections are x @ W: feeding pre-projected x with identity weights gives the same result.
    xq, xk, xv = x @ wq, x @ wk, x @ wv
    for b in range(B):
        for i in range(h):
            o = orc.diffattn_head(xq[b, :, 2 * d * i: 2 * d * i + d], xq[b, :, 2 * d * i + d: 2 * d * (i + 1)],
                                  xk[b, :, 2 * d * i: 2 * d * i + d], xk[b, :, 2 * d * i + d: 2 * d * (i + 1)],
                                  xv[b, :, Dv * i: Dv * (i + 1)], 0.5)
            np.testing.assert_allclose(y_cat[b, :, Dv * i: Dv * (i + 1)], orc.head_rmsnorm_scale(o, 0.2),
                                       atol=1e-12)


# ------------------------------------------------------------------ the layer around the module
def test_silu_matches_library_sigmoid():
    from scipy.special import expit
    t = np.linspace(-30, 30, 2001)
    np.testing.assert_allclose(orc.silu(t), t * expit(t), rtol=1e-14, atol=1e-300)


def test_rmsnorm_rows_has_closed_form_rms():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(7, 64)) * rng.uniform(0.01, 10, size=(7, 1))
    eps = 1e-5
    y = orc.rmsnorm_rows(x, eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean(y * y, axis=1), ms / (ms + eps), rtol=1e-12)
    g = rng.uniform(0.5, 2, size=64)
    np.testing.assert_allclose(orc.rmsnorm_rows(x, eps, g), y * g, rtol=1e-14)


def test_swiglu_ffn_matches_torch_float64():
    import torch
    rng = np.random.default_rng(4)
    x, wg, wu, wd = rng.normal(size=(5, 16)), rng.normal(size=(16, 24)), rng.normal(size=(16, 24)), \
        rng.normal(size=(24, 16))
    T = lambda a: torch.from_numpy(a)
    want = (torch.nn.functional.silu(T(x) @ T(wg)) * (T(x) @ T(wu))) @ T(wd)
    np.testing.assert_allclose(orc.swiglu_ffn(x, wg, wu, wd), want.numpy(), rtol=1e-12)


def _layer_weights(rng, dm, h, d, dff):
    w = lambda *s: rng.normal(size=s) / np.sqrt(s[0])
    return dict(w_q=w(dm, 2 * d * h), w_k=w(dm, 2 * d * h), w_v=w(dm, 2 * d * h), w_o=w(2 * d * h, dm),
                w_gate=w(dm, dff), w_up=w(dm, dff), w_down=w(dff, dm))


def test_layer_residual_branches():
    """With zero output weights in both branches the layer is the identity; with only the FFN's
    output weights zero it is X + module(RMSNorm(X))."""
    rng = np.random.default_rng(5)
    dm, h, d, dff = 32, 2, 8, 48
    x = rng.normal(size=(1, 6, dm))
    w = _layer_weights(rng, dm, h, d, dff)
    zero = dict(w, w_o=np.zeros_like(w["w_o"]), w_down=np.zeros_like(w["w_down"]))
    np.testing.assert_array_equal(orc.layer_fwd(x, **zero, n_heads=h, lam=0.4, lam_init=0.2), x)
    only_attn = dict(w, w_down=np.zeros_like(w["w_down"]))
    want = x + orc.module_fwd(orc.rmsnorm_rows(x), w["w_q"], w["w_k"], w["w_v"], w["w_o"], h, 0.4, 0.2)
    np.testing.assert_allclose(orc.layer_fwd(x, **only_attn, n_heads=h, lam=0.4, lam_init=0.2), want, rtol=1e-13)


def test_layer_ffn_branch_matches_torch_rms_norm():
    """With the attention output weights zero, the layer is X + FFN(RMSNorm(X)); RMSNorm and
    the FFN evaluated with torch's own float64 rms_norm and silu."""
    import torch
    F = torch.nn.functional
    rng = np.random.default_rng(6)
    dm, h, d, dff = 32, 2, 8, 48
    x = rng.normal(size=(2, 5, dm))
    w = _layer_weights(rng, dm, h, d, dff)
    g2 = rng.uniform(0.5, 1.5, size=dm)
    got = orc.layer_fwd(x, **dict(w, w_o=np.zeros_like(w["w_o"])), n_heads=h, lam=0.4, lam_init=0.2,
                        norm2_weight=g2)
    T = lambda a: torch.from_numpy(a)
    n = F.rms_norm(T(x), (dm,), T(g2), eps=1e-5)
    want = T(x) + (F.silu(n @ T(w["w_gate"])) * (n @ T(w["w_up"]))) @ T(w["w_down"])
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------- backward ---
# The pages print no gradient; the oracle's backward is pinned by central finite
# differences of its forward (a brute-force derivative of the definition), on
# shapes where every transposition changes the result (N, d and Dv all differ).

def _head_loss(q1, q2, k1, k2, v, dy, lam, lam_init, eps, w, causal):
    y = orc.head_rmsnorm_scale(orc.diffattn_head(q1, q2, k1, k2, v, lam, causal), lam_init, eps, w)
    return float(np.sum(y * dy))


def _fd(f, x, h=1e-6):
    """Central differences of the scalar f() with respect to every entry of x (in place)."""
    g = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        keep = x[idx]
        x[idx] = keep + h
        fp = f()
        x[idx] = keep - h
        fm = f()
        x[idx] = keep
        g[idx] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("causal,lam,with_w", [(True, 0.63, True), (False, -0.4, False), (True, 1.7, False)])
def test_head_backward_matches_finite_differences(causal, lam, with_w):
    r = _rng(40 + int(causal))
    N, d, Dv = 6, 4, 8
    t = {k: r.standard_normal((N, Dv if k == "v" else d)) for k in ("q1", "q2", "k1", "k2", "v")}
    dy = r.standard_normal((N, Dv))
    w = 1 + 0.3 * r.standard_normal(Dv) if with_w else None
    lam_init, eps = 0.35, 1e-5
    gr = orc.diffattn_head_bwd(t["q1"], t["q2"], t["k1"], t["k2"], t["v"], dy, lam, lam_init, eps, w, causal)
    loss = lambda: _head_loss(t["q1"], t["q2"], t["k1"], t["k2"], t["v"], dy, lam_cell[0], lam_init, eps,
                              w_cell[0], causal)
    lam_cell, w_cell = [lam], [w]
    for k in ("q1", "q2", "k1", "k2", "v"):
        np.testing.assert_allclose(gr["d" + k], _fd(loss, t[k]), rtol=1e-6, atol=1e-8, err_msg=k)
    lam_arr = np.array([lam])

    def loss_lam():
        lam_cell[0] = float(lam_arr[0])
        return loss()
    assert gr["dlam"] == pytest.approx(float(_fd(loss_lam, lam_arr)[0]), rel=1e-6, abs=1e-8)
    lam_cell[0] = lam
    w_arr = np.ones(Dv) if w is None else w.copy()

    def loss_w():
        w_cell[0] = w_arr
        return loss()
    np.testing.assert_allclose(gr["dw"], _fd(loss_w, w_arr), rtol=1e-6, atol=1e-8, err_msg="dw")


def test_head_backward_lambda_zero_is_plain_attention_backward():
    """With lambda = 0 the second map drops out: its gradients vanish and the first map's
    equal those of softmax attention followed by the same RMSNorm, which torch's float64
    autograd of scaled_dot_product_attention gives (a library routine)."""
    r = _rng(44)
    N, d, Dv = 7, 4, 6
    q1, q2, k1, k2 = (r.standard_normal((N, d)) for _ in range(4))
    v, dy = r.standard_normal((N, Dv)), r.standard_normal((N, Dv))
    gr = orc.diffattn_head_bwd(q1, q2, k1, k2, v, dy, 0.0, 0.2, 1e-5)
    assert np.all(gr["dq2"] == 0) and np.all(gr["dk2"] == 0)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q1, k1, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                                         is_causal=True)[0, 0]
    y = o / torch.sqrt((o * o).mean(-1, keepdim=True) + 1e-5) * 0.8
    (y * torch.tensor(dy)).sum().backward()
    np.testing.assert_allclose(gr["dq1"], tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gr["dk1"], tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gr["dv"], tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_batched_backward_sums_lambda_over_heads():
    r = _rng(45)
    B, H, N, d, Dv = 1, 2, 5, 4, 8
    t = {k: r.standard_normal((B, H, N, Dv if k == "v" else d)) for k in ("q1", "q2", "k1", "k2", "v")}
    dy = r.standard_normal((B, N, H, Dv))
    gr = orc.diffattn_bwd(t["q1"], t["q2"], t["k1"], t["k2"], t["v"], dy, 0.5, 0.3)
    lam_arr = np.array([0.5])
    loss = lambda: float(np.sum(orc.diffattn_fwd(t["q1"], t["q2"], t["k1"], t["k2"], t["v"], float(lam_arr[0]),
                                                 0.3) * dy))
    assert gr["dlam"] == pytest.approx(float(_fd(loss, lam_arr)[0]), rel=1e-6)
    one = orc.diffattn_head_bwd(t["q1"][0, 1], t["q2"][0, 1], t["k1"][0, 1], t["k2"][0, 1], t["v"][0, 1],
                                dy[0, :, 1, :], 0.5, 0.3)
    np.testing.assert_array_equal(gr["dk2"][0, 1], one["dk2"])


def test_reparam_lambda_backward_matches_finite_differences():
    r = _rng(46)
    vecs = [0.2 * r.standard_normal(5) for _ in range(4)]
    grads = orc.reparam_lambda_bwd(*vecs, 1.3)
    for i in range(4):
        f = lambda: 1.3 * orc.reparam_lambda(*vecs, 3)[0]
        np.testing.assert_allclose(grads[i], _fd(f, vecs[i]), rtol=1e-7, atol=1e-10)

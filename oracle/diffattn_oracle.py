"""Float64 CPU oracle for causal multi-head differential attention.

TEST INFRASTRUCTURE ONLY. This module is the plain, slow definition the GPU
library is checked against. Only the test suite, the smoke check and the
bench's CPU-baseline leg may import it; the library itself never does, and this
module imports nothing from the library.

Every function follows the definition as the source pages state it, with no
tiling, fusion or reordering beyond splitting query rows into chunks (softmax is
per row, so the split is exact):

* "Differential Transformer: Transformer que cancela ruído de atenção"
  (pt.news.hada.io), section "Como a atenção diferencial funciona":
  DiffAttn(X) = (softmax(Q1 K1^T / sqrt(d)) - lambda * softmax(Q2 K2^T / sqrt(d))) V,
  lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init,
  lambda_init = 0.8 - 0.6 * exp(-0.3 * (l - 1)); the constant 0.8 ablation.
* Same page, section "Estrutura multi-head e arquitetura completa": lambda is
  shared by the heads of one layer; each head's output gets its own RMSNorm and
  is then multiplied by (1 - lambda_init); heads are concatenated on channels
  and multiplied by W_O.
* "A Simple Principle From Noise-Cancelling Headphones Supercharges
  Transformers Like Never Before" (intoai.pub), section "A Deeper Dive Into
  Attention Calculations": the causal mask M_ij = 0 for i >= j and -inf for
  i < j; d is the query/key dimension.
* "Tag: Attention Mechanism" (priorstack.com), article "Differential
  Transformer: Canceling Context Noise with Differential Attention", section
  "Cancelling Context Noise Through Attention Map Subtraction": the same
  DiffAttn and lambda formulas in ASCII.

Readings where the pages are silent (each also listed in the design notes):
* d in sqrt(d) is the width of one query/key half.
* The same causal mask applies to both maps.
* Layer index l is 1-based, so lambda_init(1) = 0.2.
* RMSNorm: over the Dv channels of one head for one token,
  y = o / sqrt(mean(o^2) + eps) * w, eps inside the square root, w optional.
* A decode query is the last position of its sequence and sees every cached
  key, itself included.
* Module projections: Q = X W with W stored [d_in, d_out]; inside head i the
  first d channels of its 2d-wide Q (and K) slice are Q_i1, the next d are Q_i2;
  V channels [i*Dv, (i+1)*Dv) belong to head i.
* Backward pass: the pages train DIFF Transformers but print no gradient. The
  gradients here are the chain rule of the forward definition above, taken
  step by step (RMSNorm and scale, the combined map times V, the two row
  softmaxes, the two score products, lambda's reparameterisation); lambda_init
  is a constant of the layer and gets no gradient.
* Layer (intoai, "The Overall Architecture Of The Multi-Head Differential
  Transformer"; hada, "Estrutura multi-head e arquitetura completa"): the pages
  give Y = MultiHead(LN(X)) + X and X' = SwiGLU(LN(Y)) + Y with pre-RMSNorm "as
  in LLaMA". Readings: LN is RMSNorm over d_model, y = x / sqrt(mean(x^2) + eps)
  * g with eps = 1e-5 and an optional gain g; SwiGLU(x) is the LLaMA FFN
  (SiLU(x W_gate) * (x W_up)) W_down with SiLU(t) = t / (1 + e^-t).
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "lambda_init_schedule",
    "reparam_lambda",
    "causal_allowed",
    "masked_softmax_rows",
    "diffattn_head",
    "head_rmsnorm_scale",
    "diffattn_fwd",
    "diffattn_decode",
    "module_fwd",
    "rmsnorm_rows",
    "silu",
    "swiglu_ffn",
    "layer_fwd",
    "diffattn_head_bwd",
    "diffattn_bwd",
    "reparam_lambda_bwd",
]


def _f64(a) -> np.ndarray:
    """Upcast any array-like (numpy or torch CPU tensor) to a float64 ndarray."""
    if hasattr(a, "detach"):  # torch tensor: go through float32, which holds bf16 exactly
        a = a.detach().to("cpu").float().numpy()
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# lambda and lambda_init ("Como a atenção diferencial funciona")
# --------------------------------------------------------------------------

def lambda_init_schedule(layer: int) -> float:
    """lambda_init = 0.8 - 0.6 * exp(-0.3 * (l - 1)) for the 1-based layer index l."""
    if layer < 1:
        raise ValueError("layer index is 1-based")
    return 0.8 - 0.6 * math.exp(-0.3 * (layer - 1))


def reparam_lambda(lq1, lk1, lq2, lk2, layer: int, lambda_init_override: float | None = None):
    """lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init, one scalar per layer.

    Returns (lambda, lambda_init) as Python floats (float64). With
    ``lambda_init_override`` given, that constant replaces the schedule (the
    page's constant-0.8 ablation).
    """
    lq1, lk1, lq2, lk2 = (_f64(v).reshape(-1) for v in (lq1, lk1, lq2, lk2))
    if not (lq1.shape == lk1.shape == lq2.shape == lk2.shape):
        raise ValueError("lambda vectors must have one common length")
    lam_init = lambda_init_schedule(layer) if lambda_init_override is None else float(lambda_init_override)
    lam = math.exp(float(np.dot(lq1, lk1))) - math.exp(float(np.dot(lq2, lk2))) + lam_init
    return lam, lam_init


# --------------------------------------------------------------------------
# Causal mask and softmax ("A Deeper Dive Into Attention Calculations")
# --------------------------------------------------------------------------

def causal_allowed(rows: np.ndarray, n_keys: int) -> np.ndarray:
    """Boolean [len(rows), n_keys]: query position i may see key j iff i >= j."""
    j = np.arange(n_keys)[None, :]
    return np.asarray(rows)[:, None] >= j


def masked_softmax_rows(scores: np.ndarray, allowed: np.ndarray) -> np.ndarray:
    """Row softmax of scores + M, M = 0 where allowed and -inf elsewhere.

    Subtract the row max over the allowed entries, exponentiate, divide by the
    row sum. Masked entries come out exactly 0. Every row must allow at least
    one key (true for causal rows, which always see themselves).
    """
    s = np.where(allowed, scores, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=1, keepdims=True)


# --------------------------------------------------------------------------
# One head of DiffAttn ("Como a atenção diferencial funciona")
# --------------------------------------------------------------------------

def diffattn_head(q1, q2, k1, k2, v, lam: float, causal: bool = True, row_chunk: int = 512,
                  positions=None) -> np.ndarray:
    """O_hat = (softmax(Q1 K1^T/sqrt(d) + M) - lam * softmax(Q2 K2^T/sqrt(d) + M)) V.

    q1, q2: [n, d]; k1, k2: [Nk, d]; v: [Nk, Dv]. Query row r sits at position
    ``positions[r]`` (default r) and, when causal, sees keys 0..positions[r].
    Returns the pre-norm head output [n, Dv]. Query rows are processed
    ``row_chunk`` at a time.
    """
    q1, q2, k1, k2, v = (_f64(a) for a in (q1, q2, k1, k2, v))
    n, d = q1.shape
    nk = k1.shape[0]
    pos = np.arange(n) if positions is None else np.asarray(positions)
    scale = 1.0 / math.sqrt(d)
    out = np.empty((n, v.shape[1]), dtype=np.float64)
    for r0 in range(0, n, row_chunk):
        rows = np.arange(r0, min(n, r0 + row_chunk))
        allowed = causal_allowed(pos[rows], nk) if causal else np.ones((len(rows), nk), dtype=bool)
        p1 = masked_softmax_rows((q1[rows] @ k1.T) * scale, allowed)
        p2 = masked_softmax_rows((q2[rows] @ k2.T) * scale, allowed)
        out[rows] = (p1 - lam * p2) @ v
    return out


# --------------------------------------------------------------------------
# Per-head RMSNorm and the (1 - lambda_init) scale
# ("Estrutura multi-head e arquitetura completa")
# --------------------------------------------------------------------------

def head_rmsnorm_scale(o_hat, lam_init: float, eps: float = 1e-5, weight=None) -> np.ndarray:
    """y = o / sqrt(mean over Dv of o^2 + eps) * w * (1 - lambda_init), row by row."""
    o = _f64(o_hat)
    ms = np.mean(o * o, axis=-1, keepdims=True)
    y = o / np.sqrt(ms + eps)
    if weight is not None:
        y = y * _f64(weight).reshape(-1)
    return y * (1.0 - lam_init)


# --------------------------------------------------------------------------
# Batched operators matching the library's three computations
# --------------------------------------------------------------------------

def diffattn_fwd(q1, q2, k1, k2, v, lam: float, lam_init: float, eps: float = 1e-5, weight=None,
                 causal: bool = True, heads=None) -> np.ndarray:
    """Prefill: inputs [B, H, N, d] (v: [B, H, N, Dv]) -> output [B, N, H, Dv].

    The output keeps tokens outermost and heads concatenated on channels, the
    layout W_O multiplies. ``heads``, if given, is a list of (b, h) pairs to
    compute; the other output entries are NaN (used to sample big workloads).
    """
    B, H, N, _ = q1.shape
    Dv = v.shape[-1]
    out = np.full((B, N, H, Dv), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        o_hat = diffattn_head(q1[b, h], q2[b, h], k1[b, h], k2[b, h], v[b, h], lam, causal)
        out[b, :, h, :] = head_rmsnorm_scale(o_hat, lam_init, eps, weight)
    return out


def diffattn_decode(q1, q2, k1_cache, k2_cache, v_cache, seq_lens, lam: float, lam_init: float,
                    eps: float = 1e-5, weight=None, pairs=None) -> np.ndarray:
    """Decode: one new query per sequence against its KV cache.

    q1, q2: [B, H, d]; caches [B, H, Lmax, d] / [B, H, Lmax, Dv]; seq_lens: [B]
    ints (the query is the last of its sequence's L tokens and sees keys
    0..L-1). Returns [B, H, Dv]; rows not in ``pairs`` (list of (b, h)) are NaN
    when ``pairs`` is given. Written directly from the definition for a single
    query row, independently of ``diffattn_head``.
    """
    B, H, d = q1.shape[0], q1.shape[1], q1.shape[2]
    Dv = v_cache.shape[-1]
    out = np.full((B, H, Dv), np.nan)
    scale = 1.0 / math.sqrt(d)
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        L = int(seq_lens[b])
        a1 = _f64(k1_cache[b, h, :L]) @ _f64(q1[b, h]) * scale
        a2 = _f64(k2_cache[b, h, :L]) @ _f64(q2[b, h]) * scale
        p1 = np.exp(a1 - a1.max())
        p1 /= p1.sum()
        p2 = np.exp(a2 - a2.max())
        p2 /= p2.sum()
        o_hat = (p1 - lam * p2) @ _f64(v_cache[b, h, :L])
        out[b, h] = head_rmsnorm_scale(o_hat[None, :], lam_init, eps, weight)[0]
    return out


def module_fwd(x, w_q, w_k, w_v, w_o, n_heads: int, lam: float, lam_init: float, eps: float = 1e-5,
               weight=None, causal: bool = True) -> np.ndarray:
    """Multi-head differential attention module: projections, DiffAttn per head, W_O.

    x: [B, N, d_model]; w_q, w_k: [d_model, n_heads*2d]; w_v: [d_model, n_heads*Dv];
    w_o: [n_heads*Dv, d_model]. Head i reads Q_i1 = Q[..., 2di : 2di+d],
    Q_i2 = Q[..., 2di+d : 2d(i+1)] (K likewise) and V_i = V[..., i*Dv : (i+1)*Dv].
    The per-head outputs, normalised and scaled, are concatenated and multiplied
    by W_O. Returns [B, N, d_model].
    """
    x, w_q, w_k, w_v, w_o = (_f64(a) for a in (x, w_q, w_k, w_v, w_o))
    B, N, _ = x.shape
    q = x @ w_q
    k = x @ w_k
    vv = x @ w_v
    d = q.shape[-1] // (2 * n_heads)
    Dv = vv.shape[-1] // n_heads
    cat = np.empty((B, N, n_heads * Dv))
    for b in range(B):
        for i in range(n_heads):
            qs = q[b, :, 2 * d * i: 2 * d * (i + 1)]
            ks = k[b, :, 2 * d * i: 2 * d * (i + 1)]
            o_hat = diffattn_head(qs[:, :d], qs[:, d:], ks[:, :d], ks[:, d:],
                                  vv[b, :, Dv * i: Dv * (i + 1)], lam, causal)
            cat[b, :, Dv * i: Dv * (i + 1)] = head_rmsnorm_scale(o_hat, lam_init, eps, weight)
    return cat @ w_o


# --------------------------------------------------------------------------
# The layer around the module ("The Overall Architecture Of The Multi-Head
# Differential Transformer"; "Estrutura multi-head e arquitetura completa")
# --------------------------------------------------------------------------

def rmsnorm_rows(x, eps: float = 1e-5, weight=None) -> np.ndarray:
    """Pre-RMSNorm over the last axis: x / sqrt(mean(x^2) + eps), times the gain if given."""
    x = _f64(x)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return y if weight is None else y * _f64(weight).reshape(-1)


def silu(t) -> np.ndarray:
    """SiLU(t) = t / (1 + e^-t)."""
    t = _f64(t)
    return t / (1.0 + np.exp(-t))


def swiglu_ffn(x, w_gate, w_up, w_down) -> np.ndarray:
    """The LLaMA feed-forward block: (SiLU(x W_gate) * (x W_up)) W_down."""
    x, w_gate, w_up, w_down = (_f64(a) for a in (x, w_gate, w_up, w_down))
    return (silu(x @ w_gate) * (x @ w_up)) @ w_down


def layer_fwd(x, w_q, w_k, w_v, w_o, w_gate, w_up, w_down, n_heads: int, lam: float, lam_init: float,
              eps: float = 1e-5, norm1_weight=None, norm2_weight=None, head_weight=None,
              causal: bool = True) -> np.ndarray:
    """One DIFF Transformer layer: Y = MultiHead(RMSNorm(X)) + X, then SwiGLU(RMSNorm(Y)) + Y.

    x: [B, N, d_model]; the module weights as in module_fwd; w_gate, w_up: [d_model, d_ff];
    w_down: [d_ff, d_model]. The head RMSNorm uses `eps` and `head_weight`.
    """
    x = _f64(x)
    y = x + module_fwd(rmsnorm_rows(x, eps, norm1_weight), w_q, w_k, w_v, w_o, n_heads, lam, lam_init, eps,
                       head_weight, causal)
    return y + swiglu_ffn(rmsnorm_rows(y, eps, norm2_weight), w_gate, w_up, w_down)


# --------------------------------------------------------------------------
# Backward pass: the chain rule of the definition above, one step at a time
# --------------------------------------------------------------------------

def diffattn_head_bwd(q1, q2, k1, k2, v, dy, lam: float, lam_init: float, eps: float = 1e-5, weight=None,
                      causal: bool = True) -> dict:
    """Gradients of one head's y = RMSNorm((P1 - lam P2) V) * w * (1 - lam_init).

    q1, q2, k1, k2: [N, d]; v: [N, Dv]; dy: [N, Dv] (the gradient of the loss with
    respect to y). Returns dq1, dq2, dk1, dk2, dv, dlam (float) and dw ([Dv], the
    gradient with respect to the RMSNorm gain, taken as 1 when ``weight`` is None).
    Forward, with S_m = Q_m K_m^T / sqrt(d) + M and P_m its row softmax:
      A = P1 - lam P2,  O = A V,  r = sqrt(mean_c O^2 + eps),  n = O / r,  y = n w c,
    c = 1 - lam_init. Backward, row by row:
      g = dy w c;  dO = (g - n mean_c(g n)) / r;  dw = sum_rows dy n c;
      dV = A^T dO;  dA = dO V^T;  dlam = -sum(dA * P2);
      dP1 = dA,  dP2 = -lam dA;  dS_m = P_m (dP_m - rowsum(P_m dP_m));
      dQ_m = dS_m K_m / sqrt(d),  dK_m = dS_m^T Q_m / sqrt(d).
    """
    q1, q2, k1, k2, v, dy = (_f64(a) for a in (q1, q2, k1, k2, v, dy))
    n_rows, d = q1.shape
    Dv = v.shape[1]
    scale = 1.0 / math.sqrt(d)
    allowed = causal_allowed(np.arange(n_rows), k1.shape[0]) if causal else np.ones((n_rows, k1.shape[0]), bool)
    p1 = masked_softmax_rows((q1 @ k1.T) * scale, allowed)
    p2 = masked_softmax_rows((q2 @ k2.T) * scale, allowed)
    a = p1 - lam * p2
    o = a @ v
    r = np.sqrt(np.mean(o * o, axis=1, keepdims=True) + eps)
    nrm = o / r
    w = np.ones(Dv) if weight is None else _f64(weight).reshape(-1)
    c = 1.0 - lam_init
    # RMSNorm, gain and scale
    g = dy * w * c
    d_o = (g - nrm * np.mean(g * nrm, axis=1, keepdims=True)) / r
    dw = np.sum(dy * nrm * c, axis=0)
    # O = A V
    dv = a.T @ d_o
    da = d_o @ v.T
    dlam = -float(np.sum(da * p2))
    # A = P1 - lam P2, then each row softmax
    dp1, dp2 = da, -lam * da
    ds1 = p1 * (dp1 - np.sum(p1 * dp1, axis=1, keepdims=True))
    ds2 = p2 * (dp2 - np.sum(p2 * dp2, axis=1, keepdims=True))
    # S_m = Q_m K_m^T / sqrt(d)
    return {"dq1": ds1 @ k1 * scale, "dq2": ds2 @ k2 * scale, "dk1": ds1.T @ q1 * scale,
            "dk2": ds2.T @ q2 * scale, "dv": dv, "dlam": dlam, "dw": dw}


def diffattn_bwd(q1, q2, k1, k2, v, dy, lam: float, lam_init: float, eps: float = 1e-5, weight=None,
                 causal: bool = True, heads=None) -> dict:
    """Batched backward: inputs [B, H, N, d] (v [B, H, N, Dv]), dy [B, N, H, Dv] (the
    forward's output layout). Returns dq1, dq2, dk1, dk2 [B, H, N, d], dv [B, H, N, Dv],
    dlam (the sum over the heads: lambda is shared by the layer's heads) and dw [Dv].
    ``heads``, if given, lists the (b, h) pairs to compute; the other gradient entries
    are NaN and dlam, dw cover only the listed heads."""
    B, H, N, d = q1.shape
    Dv = v.shape[-1]
    out = {k: np.full((B, H, N, Dv if k == "dv" else d), np.nan) for k in ("dq1", "dq2", "dk1", "dk2", "dv")}
    dlam, dw = 0.0, np.zeros(Dv)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        gr = diffattn_head_bwd(q1[b, h], q2[b, h], k1[b, h], k2[b, h], v[b, h], _f64(dy[b, :, h, :]), lam,
                               lam_init, eps, weight, causal)
        for k in out:
            out[k][b, h] = gr[k]
        dlam += gr["dlam"]
        dw += gr["dw"]
    out["dlam"], out["dw"] = dlam, dw
    return out


def reparam_lambda_bwd(lq1, lk1, lq2, lk2, dlam: float):
    """Gradients of lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init with respect to
    the four vectors, given dlam: (dlq1, dlk1, dlq2, dlk2)."""
    lq1, lk1, lq2, lk2 = (_f64(x).reshape(-1) for x in (lq1, lk1, lq2, lk2))
    e1 = math.exp(float(np.dot(lq1, lk1)))
    e2 = math.exp(float(np.dot(lq2, lk2)))
    return dlam * e1 * lk1, dlam * e1 * lq1, -dlam * e2 * lk2, -dlam * e2 * lq2

"""Seeded synthetic inputs and the workload table.

This module holds no differential-attention arithmetic: it only draws random
tensors. The tests, the bench and the oracle-side checks all take their inputs
from here, so both sides of every comparison see the same values.

Recipe: every tensor is drawn row block by row block along its leading
dimension. Row ``b`` of tensor ``tag`` in workload ``seed`` comes from its own
``torch.Generator('cpu')`` seeded with ``sub_seed(seed, tag, b)``, as float32
``randn * std``, then rounded to bfloat16 (round-to-nearest-even) for the bf16
workloads. Any slice can therefore be regenerated alone, which is how very
large workloads are checked on sampled sequences.
"""

from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import torch

# Tensor tags: fixed so that a tensor's values never depend on which others are drawn.
TAG = {"q1": 0, "q2": 1, "k1": 2, "k2": 3, "v": 4,
       "lq1": 5, "lk1": 6, "lq2": 7, "lk2": 8,
       "x": 10, "w_q": 11, "w_k": 12, "w_v": 13, "w_o": 14, "norm_w": 15,
       "w_gate": 16, "w_up": 17, "w_down": 18, "norm1_w": 19, "norm2_w": 20, "dy": 21}


def sub_seed(seed: int, tag: int, row: int) -> int:
    return (seed * 1_000_003 + tag * 7_919 + row * 104_729 + 12_345) % (1 << 62)


def randn_rows(seed: int, tag: int, shape, std: float = 1.0, dtype=torch.bfloat16,
               rows=None, threads: int = 8) -> torch.Tensor:
    """Tensor of ``shape`` drawn row by row along dim 0 (see module docstring).

    ``rows`` restricts generation to those leading indices; the result then has
    leading size ``len(rows)`` and holds exactly those rows of the full tensor.
    """
    shape = tuple(int(s) for s in shape)
    idx = list(range(shape[0])) if rows is None else [int(r) for r in rows]
    out = torch.empty((len(idx),) + shape[1:], dtype=dtype)

    def fill(i_r):
        i, r = i_r
        g = torch.Generator().manual_seed(sub_seed(seed, tag, r))
        x = torch.randn(shape[1:], generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out[i].copy_(x.to(dtype))

    work = list(enumerate(idx))
    if threads > 1 and len(work) > 1:
        with ThreadPoolExecutor(max_workers=min(threads, len(work))) as ex:
            list(ex.map(fill, work))
    else:
        for w in work:
            fill(w)
    return out


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtype, seed and layer index."""
    name: str
    kind: str               # "prefill", "decode", "module" or "layer"
    B: int
    H: int
    N: int                  # query length (prefill/module) or cache length L (decode)
    d: int                  # width of one query/key half
    Dv: int                 # value head width
    dtype: str              # "f32" or "bf16"
    seed: int
    layer: int
    d_model: int = 0        # module and layer only
    d_ff: int = 0           # layer only: the SwiGLU hidden width
    eps: float = 1e-5
    lam_std: float = 0.1
    layers: tuple = field(default=())   # module sweep

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", "prefill", B=1, H=2, N=64, d=32, Dv=64, dtype="f32", seed=1, layer=1),
    "prefill_bf16": Workload("prefill_bf16", "prefill", B=4, H=16, N=2048, d=64, Dv=128, dtype="bf16", seed=2, layer=6),
    "long_prefill_bf16": Workload("long_prefill_bf16", "prefill", B=1, H=16, N=16384, d=64, Dv=128, dtype="bf16",
                                  seed=3, layer=12),
    "decode_bf16": Workload("decode_bf16", "decode", B=64, H=16, N=8192, d=64, Dv=128, dtype="bf16", seed=4, layer=3),
    "module_bf16": Workload("module_bf16", "module", B=2, H=8, N=4096, d=128, Dv=256, dtype="bf16", seed=5,
                            layer=1, d_model=2048, layers=tuple(range(1, 25))),
    "layer_bf16": Workload("layer_bf16", "layer", B=2, H=8, N=4096, d=128, Dv=256, dtype="bf16", seed=6, layer=1,
                           d_model=2048, d_ff=5632),
    "layer_small_bf16": Workload("layer_small_bf16", "layer", B=1, H=2, N=256, d=128, Dv=256, dtype="bf16", seed=7,
                                 layer=4, d_model=512, d_ff=1536),
}


def lambda_vectors(w: Workload):
    """The four lambda vectors (length d, float32, std ``lam_std``), drawn as one-row tensors."""
    return {k: randn_rows(w.seed, TAG[k], (1, w.d), std=w.lam_std, dtype=torch.float32)[0]
            for k in ("lq1", "lk1", "lq2", "lk2")}


def prefill_inputs(w: Workload, B=None, H=None, N=None, batch_rows=None):
    """q1, q2, k1, k2 [B,H,N,d] and v [B,H,N,Dv] as CPU tensors of the workload dtype.

    B/H/N override the workload sizes (for reduced parity cases); ``batch_rows``
    draws only those batch entries of the full tensors.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    t = {}
    for name, width in (("q1", w.d), ("q2", w.d), ("k1", w.d), ("k2", w.d), ("v", w.Dv)):
        t[name] = randn_rows(w.seed, TAG[name], (B, H, N, width), dtype=w.torch_dtype, rows=batch_rows)
    return t


def decode_inputs(w: Workload, B=None, L=None, batch_rows=None):
    """q1, q2 [B,H,d] and caches k1, k2 [B,H,L,d], v [B,H,L,Dv] (CPU, workload dtype)."""
    B = w.B if B is None else B
    L = w.N if L is None else L
    t = {}
    for name, shape in (("q1", (B, w.H, w.d)), ("q2", (B, w.H, w.d)),
                        ("k1", (B, w.H, L, w.d)), ("k2", (B, w.H, L, w.d)), ("v", (B, w.H, L, w.Dv))):
        t[name] = randn_rows(w.seed, TAG[name], shape, dtype=w.torch_dtype, rows=batch_rows)
    return t


def module_inputs(w: Workload, B=None, N=None):
    """x [B,N,d_model] ~ N(0,1) and weights [d_in, d_out] with variance 1/d_model."""
    B = w.B if B is None else B
    N = w.N if N is None else N
    dm = w.d_model
    wstd = 1.0 / math.sqrt(dm)
    t = {"x": randn_rows(w.seed, TAG["x"], (B, N, dm), dtype=w.torch_dtype)}
    for name, shape in (("w_q", (dm, w.H * 2 * w.d)), ("w_k", (dm, w.H * 2 * w.d)),
                        ("w_v", (dm, w.H * w.Dv)), ("w_o", (w.H * w.Dv, dm))):
        t[name] = randn_rows(w.seed, TAG[name], shape, std=wstd, dtype=w.torch_dtype)
    return t


def layer_inputs(w: Workload, B=None, N=None, norm_weights: bool = False):
    """module_inputs plus the SwiGLU weights w_gate, w_up [d_model, d_ff] (variance
    1/d_model) and w_down [d_ff, d_model] (variance 1/d_ff); with ``norm_weights`` also
    the two pre-RMSNorm gains norm1_w, norm2_w [d_model] = 1 + N(0, 0.1^2) (float32)."""
    t = module_inputs(w, B, N)
    dm, dff = w.d_model, w.d_ff
    t["w_gate"] = randn_rows(w.seed, TAG["w_gate"], (dm, dff), std=1.0 / math.sqrt(dm), dtype=w.torch_dtype)
    t["w_up"] = randn_rows(w.seed, TAG["w_up"], (dm, dff), std=1.0 / math.sqrt(dm), dtype=w.torch_dtype)
    t["w_down"] = randn_rows(w.seed, TAG["w_down"], (dff, dm), std=1.0 / math.sqrt(dff), dtype=w.torch_dtype)
    if norm_weights:
        for k in ("norm1_w", "norm2_w"):
            t[k] = 1.0 + randn_rows(w.seed, TAG[k], (1, dm), std=0.1, dtype=torch.float32)[0]
    return t


def output_grad(w: Workload, B=None, H=None, N=None):
    """dy [B, N, H, Dv] ~ N(0, 1): the gradient fed to the backward pass, in the prefill
    output layout and the workload dtype."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    return randn_rows(w.seed, TAG["dy"], (B, N, H, w.Dv), dtype=w.torch_dtype)

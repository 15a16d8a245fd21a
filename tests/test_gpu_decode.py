"""GPU parity of diffattn_decode against the float64 oracle."""

import numpy as np
import pytest
import torch

import differential_attention_02_gb300 as da
from differential_attention_02_gb300 import inputs as gi
from oracle import diffattn_oracle as orc
from parity import assert_bf16_parity

pytestmark = pytest.mark.gpu
NAMES = ("q1", "q2", "k1", "k2", "v")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from differential_attention_02_gb300 import build
    build.build()
    da.load_library()


def _lam(w):
    lv = gi.lambda_vectors(w)
    return orc.reparam_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer)


def _run(t, lam, lam_init, seq_lens=None, **kw):
    ws = da.workspace(da.decode_workspace_bytes(t["q1"].shape[0], t["q1"].shape[1], t["k1"].shape[2],
                                                t["q1"].shape[2], t["v"].shape[3], kw.get("num_splits", 0)))
    sl = None if seq_lens is None else torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    out = da.diffattn_decode(*(t[k].cuda() for k in NAMES), lam, lam_init, seq_lens=sl, ws=ws, **kw)
    assert da.read_error(ws) == 0
    return out


@pytest.mark.parametrize("B,L", [(1, 1), (2, 63), (3, 64), (2, 700), (1, 5000)])
def test_decode_small(B, L):
    w = gi.WORKLOADS["decode_bf16"]
    t = gi.decode_inputs(w, B=B, L=L)
    lam, lam_init = _lam(w)
    ref = orc.diffattn_decode(*(t[k] for k in NAMES), [L] * B, lam, lam_init, w.eps)
    assert_bf16_parity(_run(t, lam, lam_init), ref, f"decode B{B} L{L}")


def test_decode_ragged_lengths_ignore_stale_cache():
    w = gi.WORKLOADS["decode_bf16"]
    B, L = 4, 1000
    t = gi.decode_inputs(w, B=B, L=L)
    lens = [1000, 1, 333, 64]
    for b, n in enumerate(lens):  # entries past each length hold garbage that must not be read
        for k in ("k1", "k2", "v"):
            t[k][b, :, n:] = float("nan")
    lam, lam_init = _lam(w)
    ref = orc.diffattn_decode(*(t[k] for k in NAMES), lens, lam, lam_init, w.eps)
    assert_bf16_parity(_run(t, lam, lam_init, seq_lens=lens), ref, "ragged")


@pytest.mark.parametrize("S", [1, 2, 3, 8, 16])
def test_decode_split_count_invariance(S):
    w = gi.WORKLOADS["decode_bf16"]
    t = gi.decode_inputs(w, B=2, L=2048)
    lam, lam_init = _lam(w)
    base = _run(t, lam, lam_init, num_splits=1)
    other = _run(t, lam, lam_init, num_splits=S)
    assert float((base - other).abs().max()) < 2e-5
    ref = orc.diffattn_decode(*(t[k] for k in NAMES), [2048, 2048], lam, lam_init, w.eps)
    assert_bf16_parity(other, ref, f"S={S}")


def test_decode_wide_heads_and_bf16_out():
    g = torch.Generator().manual_seed(9)
    B, H, L, d, Dv = 2, 3, 600, 128, 256
    t = {"q1": torch.randn(B, H, d, generator=g), "q2": torch.randn(B, H, d, generator=g),
         "k1": torch.randn(B, H, L, d, generator=g), "k2": torch.randn(B, H, L, d, generator=g),
         "v": torch.randn(B, H, L, Dv, generator=g)}
    t = {k: x.to(torch.bfloat16) for k, x in t.items()}
    nw = torch.linspace(0.5, 1.5, Dv)
    ref = orc.diffattn_decode(*(t[k] for k in NAMES), [L] * B, 0.4, 0.3, 1e-5, weight=nw.numpy())
    assert_bf16_parity(_run(t, 0.4, 0.3, norm_weight=nw.cuda()), ref, "d128")
    assert_bf16_parity(_run(t, 0.4, 0.3, norm_weight=nw.cuda(), out_dtype=torch.bfloat16), ref, "d128 bf16 out")


def test_decode_matches_prefill_last_row():
    w = gi.WORKLOADS["prefill_bf16"]
    N = 777
    t = gi.prefill_inputs(w, B=1, H=4, N=N)
    lam, lam_init = 0.55, 0.47
    pre = da.diffattn_fwd(*(t[k].cuda() for k in NAMES), lam, lam_init)
    dec_in = {"q1": t["q1"][:, :, -1].contiguous(), "q2": t["q2"][:, :, -1].contiguous(), "k1": t["k1"],
              "k2": t["k2"], "v": t["v"]}
    dec = _run(dec_in, lam, lam_init)
    assert float((pre[:, -1] - dec).abs().max()) < 5e-3


def test_decode_workload_sampled_sequences():
    """64 sequences x 16 heads x 8192 cached tokens; oracle on 6 sampled sequences, all heads."""
    w = gi.WORKLOADS["decode_bf16"]
    t = gi.decode_inputs(w)
    lam, lam_init = _lam(w)
    out = _run(t, lam, lam_init)
    seqs = [0, 5, 17, 31, 48, 63]
    ref = np.full(out.shape, np.nan)
    r = orc.diffattn_decode(*(t[k][seqs] for k in NAMES), [w.N] * len(seqs), lam, lam_init, w.eps)
    ref[seqs] = r
    assert_bf16_parity(out, ref, "decode workload")

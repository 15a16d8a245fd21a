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


# ------------------------------------------------------------------ paged KV cache, shared KV heads
def _paged(cache, lens, page=64, spare=5, seed=0):
    """Scatters a contiguous cache [B, Hk, L, w] into a shuffled pool of pages [P, Hk, page, w]
    and returns (pool, block_table [B, max_pages])."""
    B, Hk, L, w = cache.shape
    maxp = (L + page - 1) // page
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(B * maxp + spare, generator=g)[: B * maxp].view(B, maxp)
    pool = torch.zeros(B * maxp + spare, Hk, page, w, dtype=cache.dtype)
    for b in range(B):
        for i in range(maxp):
            rows = cache[b, :, i * page: min(L, (i + 1) * page)]
            pool[perm[b, i], :, : rows.shape[1]] = rows
    return pool, perm.to(torch.int32)


def test_paged_decode_matches_contiguous_and_oracle():
    w = gi.WORKLOADS["decode_bf16"]
    B, L = 3, 1000
    host = gi.decode_inputs(w, B=B, L=L)
    lens_l = [1000, 77, 640]
    lens = torch.tensor(lens_l, dtype=torch.int32, device="cuda")
    t = {k: host[k].cuda() for k in NAMES}
    lam, lam_init = 0.45, 0.47
    want = da.diffattn_decode(*(t[k] for k in NAMES), lam, lam_init, seq_lens=lens)
    pools = {}
    for k in ("k1", "k2", "v"):
        pools[k], table = _paged(host[k], lens_l)
    got = da.diffattn_decode_paged(t["q1"], t["q2"], pools["k1"].cuda(), pools["k2"].cuda(), pools["v"].cuda(),
                                   table.cuda(), lens, lam, lam_init, L=L)
    torch.cuda.synchronize()
    assert torch.equal(got, want)  # the same kernels, split geometry and values
    ref = orc.diffattn_decode(host["q1"], host["q2"], host["k1"], host["k2"], host["v"], lens_l, lam, lam_init)
    assert_bf16_parity(got, ref, "paged decode")


def test_paged_decode_grouped_kv_heads():
    """H query heads read H / kv_group KV heads: equal to the decode on KV heads expanded to H."""
    g = torch.Generator().manual_seed(21)
    B, H, group, L, d, Dv = 2, 4, 2, 300, 64, 128
    q1, q2 = (torch.randn(B, H, d, generator=g).to(torch.bfloat16) for _ in range(2))
    k1, k2 = (torch.randn(B, H // group, L, d, generator=g).to(torch.bfloat16) for _ in range(2))
    v = torch.randn(B, H // group, L, Dv, generator=g).to(torch.bfloat16)
    lens_l = [300, 129]
    lens = torch.tensor(lens_l, dtype=torch.int32, device="cuda")
    expand = lambda x: x.repeat_interleave(group, dim=1)  # query head h reads KV head h // group
    lam, lam_init = 0.6, 0.2
    want = da.diffattn_decode(q1.cuda(), q2.cuda(), expand(k1).cuda(), expand(k2).cuda(), expand(v).cuda(), lam,
                              lam_init, seq_lens=lens)
    p1, table = _paged(k1, lens_l, seed=3)
    p2, _ = _paged(k2, lens_l, seed=3)
    pv, _ = _paged(v, lens_l, seed=3)
    got = da.diffattn_decode_paged(q1.cuda(), q2.cuda(), p1.cuda(), p2.cuda(), pv.cuda(), table.cuda(), lens, lam,
                                   lam_init, L=L, kv_group=group)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    ref = orc.diffattn_decode(q1, q2, expand(k1), expand(k2), expand(v), lens_l, lam, lam_init)
    assert_bf16_parity(got, ref, "grouped paged decode")


def test_kv_append_paged_then_decode():
    """Appending the new token with diffattn_kv_append_paged writes exactly the expected rows
    (bit-exact against a host scatter), and the decode that follows equals the contiguous
    decode over a cache that already holds that token."""
    w = gi.WORKLOADS["decode_bf16"]
    B, L = 3, 704
    host = gi.decode_inputs(w, B=B, L=L)
    lens_l = [704, 65, 131]  # the new token at position len - 1: a page's last row, a fresh page, mid-page
    lens = torch.tensor(lens_l, dtype=torch.int32, device="cuda")
    pools, table = {}, None
    for k in ("k1", "k2", "v"):
        c = host[k].clone()
        for b, n in enumerate(lens_l):
            c[b, :, n - 1] = 0  # the token to be appended is not in the cache yet
        pools[k], table = _paged(c, lens_l, seed=9)
    new = {k: torch.stack([host[k][b, :, n - 1] for b, n in enumerate(lens_l)]) for k in ("k1", "k2", "v")}
    dev_pools = {k: pools[k].cuda() for k in pools}
    da.diffattn_kv_append_paged(new["k1"].cuda(), new["k2"].cuda(), new["v"].cuda(), dev_pools["k1"],
                                dev_pools["k2"], dev_pools["v"], table.cuda(), lens)
    torch.cuda.synchronize()
    for k in pools:
        want = pools[k].clone()
        for b, n in enumerate(lens_l):
            want[table[b, (n - 1) // 64], :, (n - 1) % 64] = new[k][b]
        assert torch.equal(dev_pools[k].cpu(), want), k
    t = {k: host[k].cuda() for k in NAMES}
    lam, lam_init = 0.45, 0.47
    want = da.diffattn_decode(*(t[k] for k in NAMES), lam, lam_init, seq_lens=lens)
    got = da.diffattn_decode_paged(t["q1"], t["q2"], dev_pools["k1"], dev_pools["k2"], dev_pools["v"],
                                   table.cuda(), lens, lam, lam_init, L=L)
    torch.cuda.synchronize()
    assert torch.equal(got, want)

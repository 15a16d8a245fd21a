"""GPU checks of the serving decode over an fp8 (e4m3) KV cache.

The decode reads e4m3 bytes and one scale per tensor. Its dot products are exact
f16 x f16 products (every e4m3 value is an f16 value; the query is held as f16
scaled by a power of two) accumulated in fp32, and the softmax weights are
rounded to f16 for the P.V products (a relative 2^-11, as the prefill rounds P),
so it is compared with the float64 oracle run on exactly the dequantized values,
at the bar of the bf16 decode. The append must quantize like a plain
round-to-nearest-even cast of x / scale."""

import numpy as np
import pytest
import torch

import differential_attention_02_gb300 as da
from differential_attention_02_gb300 import inputs as gi
from oracle import diffattn_oracle as orc
from parity import assert_bf16_parity

pytestmark = pytest.mark.gpu
F8 = torch.float8_e4m3fn


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from differential_attention_02_gb300 import build
    build.build()
    da.load_library()


def _quant(x, scale):
    return (x.float() / scale).to(F8)


def _paged(cache, page=64, spare=3, seed=0):
    """Scatter [B, Hk, L, w] into a shuffled pool [P, Hk, page, w]; returns (pool, table)."""
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


@pytest.mark.parametrize("d,Dv,group", [(64, 128, 1), (128, 256, 1), (64, 128, 2)])
def test_fp8_paged_decode_matches_oracle_on_dequantized_cache(d, Dv, group):
    g = torch.Generator().manual_seed(d + group)
    B, H, L = 3, 4, 1000
    Hk = H // group
    q1, q2 = (torch.randn(B, H, d, generator=g).to(torch.bfloat16) for _ in range(2))
    kv = {"k1": torch.randn(B, Hk, L, d, generator=g), "k2": torch.randn(B, Hk, L, d, generator=g),
          "v": torch.randn(B, Hk, L, Dv, generator=g)}
    scales = tuple(float(kv[k].abs().max()) / 448.0 for k in ("k1", "k2", "v"))
    q8 = {k: _quant(kv[k], s) for k, s in zip(("k1", "k2", "v"), scales)}
    deq = {k: q8[k].float() * s for k, s in zip(("k1", "k2", "v"), scales)}
    lens_l = [1000, 77, 640]
    lens = torch.tensor(lens_l, dtype=torch.int32, device="cuda")
    pools, table = {}, None
    for k in q8:
        pools[k], table = _paged(q8[k], seed=5)
    lam, lam_init = 0.45, 0.47
    got = da.diffattn_decode_paged(q1.cuda(), q2.cuda(), pools["k1"].cuda(), pools["k2"].cuda(), pools["v"].cuda(),
                                   table.cuda(), lens, lam, lam_init, L=L, kv_group=group, scales=scales)
    torch.cuda.synchronize()
    expand = lambda x: x.repeat_interleave(group, dim=1)
    ref = orc.diffattn_decode(q1, q2, expand(deq["k1"]), expand(deq["k2"]), expand(deq["v"]), lens_l, lam, lam_init)
    assert_bf16_parity(got, ref, f"fp8 paged decode d{d} group{group}")


@pytest.mark.parametrize("q_scale", [1e-5, 3e4])
def test_fp8_decode_query_magnitudes(q_scale):
    """Queries far from unit scale: 1e-5 (f16 subnormal range without the power-of-two
    scaling) and 3e4 (elements past the f16 limit of 65504). Scores of order q_scale
    give a flat softmax at 1e-5 and a nearly one-hot one at 3e4; both meet the oracle."""
    g = torch.Generator().manual_seed(31)
    B, H, L, d, Dv = 2, 3, 700, 64, 128
    q1, q2 = ((torch.randn(B, H, d, generator=g) * q_scale).to(torch.bfloat16) for _ in range(2))
    kv = {"k1": torch.randn(B, H, L, d, generator=g), "k2": torch.randn(B, H, L, d, generator=g),
          "v": torch.randn(B, H, L, Dv, generator=g)}
    scales = tuple(float(kv[k].abs().max()) / 448.0 for k in ("k1", "k2", "v"))
    q8 = {k: _quant(kv[k], s) for k, s in zip(("k1", "k2", "v"), scales)}
    deq = {k: q8[k].float() * s for k, s in zip(("k1", "k2", "v"), scales)}
    lens_l = [700, 333]
    lens = torch.tensor(lens_l, dtype=torch.int32, device="cuda")
    pools, table = {}, None
    for k in q8:
        pools[k], table = _paged(q8[k], seed=8)
    got = da.diffattn_decode_paged(q1.cuda(), q2.cuda(), pools["k1"].cuda(), pools["k2"].cuda(), pools["v"].cuda(),
                                   table.cuda(), lens, 0.6, 0.3, L=L, scales=scales)
    torch.cuda.synchronize()
    ref = orc.diffattn_decode(q1, q2, deq["k1"], deq["k2"], deq["v"], lens_l, 0.6, 0.3)
    assert_bf16_parity(got, ref, f"fp8 decode, queries x {q_scale}")


def test_fp8_append_quantizes_like_a_cast_and_saturates():
    g = torch.Generator().manual_seed(77)
    B, Hk, d, Dv, L = 3, 2, 64, 128, 200
    lens_l = [200, 65, 1]
    lens = torch.tensor(lens_l, dtype=torch.int32, device="cuda")
    scales = (0.011, 0.013, 0.017)
    pools, table = {}, None
    for k, w in (("k1", d), ("k2", d), ("v", Dv)):
        pools[k], table = _paged(torch.zeros(B, Hk, L, w, dtype=F8), seed=2)
    new = {k: (torch.randn(B, Hk, w, generator=g) * 2).to(torch.bfloat16) for k, w in (("k1", d), ("k2", d), ("v", Dv))}
    new["k1"][0, 0, :4] = torch.tensor([1e4, -1e4, 5.0, -5.0], dtype=torch.bfloat16)  # beyond 448 * scale
    dev = {k: pools[k].cuda() for k in pools}
    da.diffattn_kv_append_paged(new["k1"].cuda(), new["k2"].cuda(), new["v"].cuda(), dev["k1"], dev["k2"], dev["v"],
                                table.cuda(), lens, scales=scales)
    torch.cuda.synchronize()
    for k, s in zip(("k1", "k2", "v"), scales):
        want = pools[k].clone()
        for b, n in enumerate(lens_l):
            want[table[b, (n - 1) // 64], :, (n - 1) % 64] = _quant(new[k][b].float().clamp(-448 * s, 448 * s), s)
        assert torch.equal(dev[k].cpu().view(torch.uint8), want.view(torch.uint8)), k
    row = dev["k1"].cpu()[table[0, (lens_l[0] - 1) // 64], 0, (lens_l[0] - 1) % 64, :2].view(torch.uint8)
    assert row.tolist() == [0x7E, 0xFE]  # +448 and -448, the largest finite e4m3 values


def test_fp8_append_then_decode_equals_decode_of_the_filled_cache():
    w = gi.WORKLOADS["decode_bf16"]
    B, L = 2, 300
    host = gi.decode_inputs(w, B=B, L=L)
    lens_l = [300, 129]
    lens = torch.tensor(lens_l, dtype=torch.int32, device="cuda")
    scales = tuple(float(host[k].float().abs().max()) / 448.0 for k in ("k1", "k2", "v"))
    full, holed, table = {}, {}, None
    for k, s in zip(("k1", "k2", "v"), scales):
        q = _quant(host[k], s)
        h = q.clone()
        for b, n in enumerate(lens_l):
            h[b, :, n - 1] = _quant(torch.zeros(1), 1.0)
        full[k], table = _paged(q, seed=4)
        holed[k], _ = _paged(h, seed=4)
    new = {k: torch.stack([host[k][b, :, n - 1] for b, n in enumerate(lens_l)]).contiguous() for k in ("k1", "k2", "v")}
    dh = {k: holed[k].cuda() for k in holed}
    da.diffattn_kv_append_paged(new["k1"].cuda(), new["k2"].cuda(), new["v"].cuda(), dh["k1"], dh["k2"], dh["v"],
                                table.cuda(), lens, scales=scales)
    q1, q2 = host["q1"].cuda(), host["q2"].cuda()
    args = (table.cuda(), lens, 0.5, 0.3)
    got = da.diffattn_decode_paged(q1, q2, dh["k1"], dh["k2"], dh["v"], *args, L=L, scales=scales)
    want = da.diffattn_decode_paged(q1, q2, full["k1"].cuda(), full["k2"].cuda(), full["v"].cuda(), *args, L=L,
                                    scales=scales)
    torch.cuda.synchronize()
    assert torch.equal(got, want)

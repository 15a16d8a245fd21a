"""The seeded generators: deterministic, sliceable, and with the stated distributions."""

import math

import torch

from differential_attention_02_gb300 import inputs as gi


def test_rows_regenerate_exactly_and_are_deterministic():
    full = gi.randn_rows(7, gi.TAG["k1"], (5, 3, 9, 4))
    part = gi.randn_rows(7, gi.TAG["k1"], (5, 3, 9, 4), rows=[3, 1])
    assert torch.equal(part[0], full[3]) and torch.equal(part[1], full[1])
    again = gi.randn_rows(7, gi.TAG["k1"], (5, 3, 9, 4), threads=1)
    assert torch.equal(full, again)
    other = gi.randn_rows(7, gi.TAG["k2"], (5, 3, 9, 4))
    assert not torch.equal(full, other)


def test_bf16_values_are_rounded_float32_draws():
    x = gi.randn_rows(3, 0, (2, 1000), dtype=torch.bfloat16)
    f = gi.randn_rows(3, 0, (2, 1000), dtype=torch.float32)
    assert torch.equal(x, f.to(torch.bfloat16))


def test_workload_distributions():
    w = gi.WORKLOADS["module_bf16"]
    wq = gi.randn_rows(w.seed, gi.TAG["w_q"], (256, 2048), std=1 / math.sqrt(w.d_model), dtype=torch.float32)
    assert abs(wq.var().item() - 1 / 2048) < 0.05 / 2048
    lv = gi.lambda_vectors(gi.WORKLOADS["tiny_fp32"])
    assert set(lv) == {"lq1", "lk1", "lq2", "lk2"} and lv["lq1"].shape == (32,)
    t = gi.prefill_inputs(gi.WORKLOADS["tiny_fp32"])
    assert t["q1"].shape == (1, 2, 64, 32) and t["v"].shape == (1, 2, 64, 64) and t["q1"].dtype == torch.float32

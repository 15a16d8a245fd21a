"""GPU parity of the multi-head differential attention module (three projection
GEMMs, fused attention on strided views, W_O GEMM) against the float64 oracle."""

import numpy as np
import pytest
import torch

import differential_attention_02_gb300 as da
from differential_attention_02_gb300 import inputs as gi
from oracle import diffattn_oracle as orc
from parity import assert_bf16_parity, errors

pytestmark = pytest.mark.gpu
W = gi.WORKLOADS["module_bf16"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from differential_attention_02_gb300 import build
    build.build()
    da.load_library()


def _lam(layer):
    lv = gi.lambda_vectors(W)
    return orc.reparam_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], layer)


def _module(t, layer, fused_qkv=False):
    lam, lam_init = _lam(layer)
    dev = {k: v.cuda() for k, v in t.items()}
    ws = da.workspace(256)
    wqkv = torch.cat([dev["w_q"], dev["w_k"], dev["w_v"]], dim=1).contiguous() if fused_qkv else None
    y = da.module_fwd(dev["x"], dev["w_q"], dev["w_k"], dev["w_v"], dev["w_o"], W.H, lam, lam_init, W.eps, ws=ws,
                      out_dtype=torch.float32, w_qkv=wqkv)
    assert da.read_error(ws) == 0
    ref = orc.module_fwd(t["x"], t["w_q"], t["w_k"], t["w_v"], t["w_o"], W.H, lam, lam_init, W.eps)
    return y, ref


@pytest.mark.parametrize("layer,fused_qkv", [(1, False), (7, False), (24, False), (7, True)])
def test_module_reduced_length(layer, fused_qkv):
    """N = 512, three layers; the projections as three GEMMs or one against [W_Q | W_K | W_V]
    (Q, K, V then column blocks of one output, read in place with its row stride)."""
    t = gi.module_inputs(W, B=1, N=512)
    y, ref = _module(t, layer, fused_qkv)
    ma, rr = errors(y, ref)
    print(f"layer {layer}: max-abs {ma:.3e} rel-RMS {rr:.3e}")
    assert_bf16_parity(y, ref, f"module N=512 layer {layer}")


def test_module_workload_full():
    """X [2, 4096, 2048], h=8, d=128, Dv=256, layer 1: every output element."""
    t = gi.module_inputs(W)
    y, ref = _module(t, 1, fused_qkv=True)
    ma, rr = errors(y, ref)
    print(f"module workload: max-abs {ma:.3e} rel-RMS {rr:.3e}")
    assert_bf16_parity(y, ref, "module workload")

"""Failure detection on the GPU without a fault: a wait that can never complete
gives up after its bound, the error is reported through the workspace, and
the context stays usable for the next call."""

import ctypes
import time

import pytest
import torch

import differential_attention_02_gb300 as da
from differential_attention_02_gb300 import inputs as gi
from oracle import diffattn_oracle as orc
from parity import assert_bf16_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from differential_attention_02_gb300 import build
    build.build()
    return da.load_library()


def test_bounded_wait_reports_timeout_and_context_survives(lib):
    ws = torch.zeros(512, dtype=torch.uint8, device="cuda")
    ws = ws[(-ws.data_ptr()) % 256:]
    t0 = time.time()
    st = lib.diffattn_selftest_timeout(ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == da.OK
    code = da.read_error(ws)
    elapsed = time.time() - t0
    assert code == (0x7F << 8) | 1
    assert 0.5 < elapsed < 30.0, elapsed
    assert da.read_error(ws) == 0  # cleared by the first read
    # the context still works: a normal call afterwards is correct
    w = gi.WORKLOADS["prefill_bf16"]
    t = gi.prefill_inputs(w, B=1, H=1, N=130)
    ref = orc.diffattn_fwd(*(t[k] for k in ("q1", "q2", "k1", "k2", "v")), 0.4, 0.3)
    out = da.diffattn_fwd(*(t[k].cuda() for k in ("q1", "q2", "k1", "k2", "v")), 0.4, 0.3, ws=ws)
    assert da.read_error(ws) == 0
    assert_bf16_parity(out, ref, "after timeout")

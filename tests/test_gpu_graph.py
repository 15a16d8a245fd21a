"""CUDA-graph capture of the library's multi-launch paths.

Training and serving loops capture steps into CUDA graphs. The paths checked here
enqueue more than one launch: the module (three kernels chained as programmatic
dependent launches) and the training pair's backward (the preparation, the key side
as a dependent launch, the query side and the reduction on a library side stream
forked and joined with events). Each is captured after one eager call (which sets
up the workspace and the side stream), replayed twice, and must reproduce the eager
results bit for bit: every path is deterministic, so any difference would be an
ordering error in the captured graph.
"""

import pytest
import torch

import differential_attention_02_gb300 as da
from differential_attention_02_gb300 import inputs as gi

pytestmark = pytest.mark.gpu
NAMES = ("q1", "q2", "k1", "k2", "v")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from differential_attention_02_gb300 import build
    build.build()
    da.load_library()


def _replay_twice(fn):
    """Captures fn() on a side stream, replays the graph twice, returns its outputs."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up on the capture stream (library streams and workspaces exist after it)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    return out


def test_graph_prefill():
    w = gi.WORKLOADS["prefill_bf16"]
    t = {k: v.cuda() for k, v in gi.prefill_inputs(w, B=2, H=4, N=640).items()}
    ws = da.workspace(256)
    fn = lambda: da.diffattn_fwd(*(t[k] for k in NAMES), 0.6, 0.8, w.eps, out_dtype=torch.bfloat16, ws=ws)
    ref = fn().clone()
    got = _replay_twice(fn)
    assert da.read_error(ws) == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_graph_module():
    w = gi.WORKLOADS["module_bf16"]
    t = {k: v.cuda() for k, v in gi.module_inputs(w, N=512).items()}
    ws = da.workspace(256)
    fn = lambda: da.module_fwd(t["x"], t["w_q"], t["w_k"], t["w_v"], t["w_o"], w.H, 0.6, 0.8, w.eps, ws=ws,
                               out_dtype=torch.float32)
    ref = fn().clone()
    got = _replay_twice(fn)
    assert da.read_error(ws) == 0
    assert torch.equal(got, ref)


def test_graph_training_pair_backward():
    w = gi.WORKLOADS["prefill_bf16"]
    B, H, N = 2, 4, 640
    t = {k: v.cuda() for k, v in gi.prefill_inputs(w, B=B, H=H, N=N).items()}
    dy = (torch.randn(B, N, H, w.Dv, generator=torch.Generator().manual_seed(5))).to(torch.bfloat16).cuda()
    nw = torch.linspace(0.5, 1.5, w.Dv).cuda()
    _, saved = da.diffattn_fwd_train(*(t[k] for k in NAMES), 0.6, 0.8, w.eps, norm_weight=nw,
                                     out_dtype=torch.bfloat16)
    ws = da.workspace(da.bwd_workspace_bytes(B, H, N, w.d, w.Dv))
    fn = lambda: da.diffattn_bwd(*(t[k] for k in NAMES), dy, 0.6, 0.8, w.eps, norm_weight=nw, want_dnorm_weight=True,
                                 ws=ws, saved=saved)
    ref = {k: v.clone() for k, v in fn().items()}
    got = _replay_twice(fn)
    assert da.read_error(ws) == 0
    for k in ("dq1", "dq2", "dk1", "dk2", "dv", "dlam", "dw"):
        assert torch.equal(got[k], ref[k]), k

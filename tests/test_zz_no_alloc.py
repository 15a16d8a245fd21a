"""diffattn_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (no workspace argument; the library's own fixed-size
scratch holds the split partial states). Checked through the C ABI against
diffattn_decode, which uses a caller workspace, on two calls in a row; the
second call is also checked to allocate nothing, and the scratch's error word
is read back through its accessor."""

import ctypes

import pytest
import torch

import differential_attention_02_gb300 as da
from differential_attention_02_gb300 import inputs as gi
from parity import assert_bf16_parity

pytestmark = pytest.mark.gpu
NAMES = ("q1", "q2", "k1", "k2", "v")


@pytest.fixture(scope="module")
def lib():
    from differential_attention_02_gb300 import build
    build.build()
    return da.load_library()


def _noalloc(lib, t, lam, lam_init, seq_lens=None, num_splits=0, out=None):
    B, H, d = t["q1"].shape
    Dv = t["v"].shape[-1]
    L = t["k1"].shape[2]
    if out is None:
        out = torch.full((B, H, Dv), float("nan"), dtype=torch.float32, device="cuda")
    sl = None if seq_lens is None else ctypes.c_void_p(seq_lens.data_ptr())
    st = lib.diffattn_decode_noalloc(
        ctypes.c_void_p(t["q1"].data_ptr()), ctypes.c_void_p(t["q2"].data_ptr()), da._t4(t["k1"]), da._t4(t["k2"]),
        da._t4(t["v"]), sl, L, ctypes.c_void_p(out.data_ptr()), None, B, H, d, Dv, lam, lam_init, 1e-5, num_splits,
        da.F32, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


def _read_error(lib):
    code = ctypes.c_int32(-1)
    st = lib.diffattn_decode_noalloc_read_error(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                                 ctypes.byref(code))
    return st, code.value


def test_noalloc_decode_matches_workspace_decode_twice(lib):
    w = gi.WORKLOADS["decode_bf16"]
    cases = [(gi.decode_inputs(w, B=3, L=1500), [1500, 7, 900], 0),   # ragged lengths, auto splits
             (gi.decode_inputs(w, B=2, L=4096), None, 4)]              # next call reuses the same scratch
    for host, lens, splits in cases:
        t = {k: host[k].cuda() for k in NAMES}
        sl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
        want = da.diffattn_decode(*(t[k] for k in NAMES), 0.45, 0.47, seq_lens=sl, num_splits=splits)
        st, got = _noalloc(lib, t, 0.45, 0.47, seq_lens=sl, num_splits=splits)
        assert st == da.OK, da.status_string(st)
        torch.cuda.synchronize()
        assert_bf16_parity(got, want.double().cpu().numpy(), "no-alloc vs workspace decode")
        assert torch.equal(got, want)  # same kernels, same split geometry
        assert _read_error(lib) == (da.OK, 0)  # no device-side wait gave up


def test_noalloc_decode_allocates_nothing(lib):
    """After a first call (which sets the library up on this device), a further call
    changes neither the driver's free device memory nor torch's allocation counts."""
    w = gi.WORKLOADS["decode_bf16"]
    host = gi.decode_inputs(w, B=2, L=2048)
    t = {k: host[k].cuda() for k in NAMES}
    out = torch.empty((2, w.H, w.Dv), dtype=torch.float32, device="cuda")
    st, _ = _noalloc(lib, t, 0.3, 0.2, out=out)
    assert st == da.OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    n0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    st, _ = _noalloc(lib, t, 0.3, 0.2, out=out)
    assert st == da.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    n1 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    assert free1 == free0
    assert n1 == n0
    want = da.diffattn_decode(*(t[k] for k in NAMES), 0.3, 0.2)
    assert torch.equal(out, want)


def test_noalloc_decode_rejects_oversized_requests(lib):
    # Views of one [L, width] buffer repeated over 64 sequences x 16 heads (zero batch and
    # head strides: valid operands, and only the scratch-size check can reject the call).
    L = 65536
    t = {"q1": torch.zeros(64, 16, 64, dtype=torch.bfloat16, device="cuda"),
         "q2": torch.zeros(64, 16, 64, dtype=torch.bfloat16, device="cuda"),
         "k1": torch.zeros(1, 1, L, 64, dtype=torch.bfloat16, device="cuda").expand(64, 16, L, 64),
         "k2": torch.zeros(1, 1, L, 64, dtype=torch.bfloat16, device="cuda").expand(64, 16, L, 64),
         "v": torch.zeros(1, 1, L, 128, dtype=torch.bfloat16, device="cuda").expand(64, 16, L, 128)}
    # 64 sequences x 16 heads x 256 splits of partial states is far beyond the 8 MiB scratch.
    need = da.decode_workspace_bytes(64, 16, L, 64, 128, 256)
    assert need > 8 << 20
    st, _ = _noalloc(lib, t, 0.5, 0.2, num_splits=256)
    assert st == da.ERR_WORKSPACE

"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the header declares, computes lambda on the host like the
oracle, and rejects bad arguments before launching anything."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

import differential_attention_02_gb300 as da
from differential_attention_02_gb300 import build as dab
from oracle import diffattn_oracle as orc

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "diffattn.h")


@pytest.fixture(scope="module")
def lib():
    dab.build()
    return da.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(diffattn_[a-z0-9_]+)\s*\(", text)))


def test_header_and_library_agree(lib):
    names = _declared_functions()
    assert set(names) == set(da.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_header_is_plain_c_and_links_against_the_library(lib, tmp_path):
    """A C99 translation unit that includes the header and takes the address of every
    declared function compiles with warnings as errors and links against the library."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = _declared_functions()
    src = tmp_path / "use_header.c"
    # Besides referencing every entry point, the program calls the host-only ones: lambda for
    # layer 1 from zero vectors is exp(0) - exp(0) + 0.2 = 0.2, and a status string.
    src.write_text('#include "diffattn.h"\n#include <stdio.h>\ntypedef void (*fn_t)(void);\n'
                   "int main(void) {\n    fn_t fns[] = {\n"
                   + "".join(f"        (fn_t)&{n},\n" for n in names)
                   + "    };\n"
                   "    float z[4] = {0.f, 0.f, 0.f, 0.f}, lam = -1.f, lam_init = -1.f;\n"
                   "    diffattn_status st = diffattn_lambda(z, z, z, z, 4, 1, -1.f, &lam, &lam_init);\n"
                   "    printf(\"%d %d %.6f %.6f %s\\n\", (int)(sizeof fns / sizeof fns[0]), (int)st, lam, lam_init,\n"
                   "           diffattn_status_string(DIFFATTN_ERR_WORKSPACE));\n"
                   "    return 0;\n}\n")
    pkg = os.path.dirname(da.__file__)
    out = tmp_path / "use_header"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.dirname(HEADER), str(src), "-o", str(out), "-L", pkg, "-ldiffattn"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    # The library carries the CUDA runtime statically: the program loads it with nothing else.
    r = subprocess.run([str(out)], capture_output=True, text=True, env={**os.environ, "LD_LIBRARY_PATH": pkg})
    assert r.returncode == 0, r.stderr
    count, status, lam, lam_init, text = r.stdout.split(maxsplit=4)
    assert int(count) == len(names) and int(status) == da.OK
    assert float(lam) == pytest.approx(0.2, abs=1e-6) and float(lam_init) == pytest.approx(0.2, abs=1e-6)
    assert text.strip() == da.status_string(da.ERR_WORKSPACE)


def test_status_strings(lib):
    assert da.status_string(da.OK) == "ok"
    assert "timed out" in da.status_string(da.ERR_TIMEOUT)
    assert da.status_string(99) == "unknown status"


@pytest.mark.parametrize("layer", [1, 2, 6, 12, 24])
def test_host_lambda_matches_oracle(lib, layer):
    rng = np.random.default_rng(layer)
    vs = [rng.normal(size=64).astype(np.float32) * 0.1 for _ in range(4)]
    lam, lam_init = da.diffattn_lambda(*vs, layer)
    lam64, lam_init64 = orc.reparam_lambda(*vs, layer)
    assert lam == pytest.approx(lam64, abs=2e-7, rel=1e-6)
    assert lam_init == pytest.approx(lam_init64, abs=1e-7)
    lam, lam_init = da.diffattn_lambda(*vs, layer, lambda_init_override=0.8)
    assert lam_init == pytest.approx(0.8, abs=1e-7)
    assert lam == pytest.approx(orc.reparam_lambda(*vs, layer, 0.8)[0], abs=2e-7)


def test_lambda_rejects_bad_arguments(lib):
    z = np.zeros(4, np.float32)
    with pytest.raises(da.DiffAttnError) as e:
        da.diffattn_lambda(z, z, z, z, 0)
    assert e.value.status == da.ERR_INVALID_ARG
    big = np.full(4, 100.0, np.float32)
    with pytest.raises(da.DiffAttnError):
        da.diffattn_lambda(big, big, z, z, 1)  # exp overflows


def _tensor(ptr=0x10000, sb=4096, sh=1024, sn=64):
    return da.Tensor4(ptr, sb, sh, sn)


def _fwd(lib, **kw):
    a = dict(q1=_tensor(), q2=_tensor(), k1=_tensor(), k2=_tensor(), v=_tensor(sn=128), out=0x20000, w=None,
             B=1, H=2, N=16, d=64, Dv=128, causal=1, lam=0.5, lam_init=0.2, eps=1e-5, ind=da.BF16, outd=da.F32,
             ws=0x40000, wsb=256, stream=None)
    a.update(kw)
    return lib.diffattn_fwd(a["q1"], a["q2"], a["k1"], a["k2"], a["v"], a["out"], a["w"], a["B"], a["H"], a["N"],
                            a["d"], a["Dv"], a["causal"], a["lam"], a["lam_init"], a["eps"], a["ind"], a["outd"],
                            a["ws"], a["wsb"], a["stream"])


def test_fwd_argument_validation(lib):
    assert _fwd(lib, B=-1) == da.ERR_INVALID_ARG
    assert _fwd(lib, B=0) == da.OK and _fwd(lib, N=0) == da.OK  # nothing to do
    assert _fwd(lib, q1=_tensor(ptr=0)) == da.ERR_INVALID_ARG
    assert _fwd(lib, k2=_tensor(ptr=0x10008)) == da.ERR_INVALID_ARG      # misaligned
    assert _fwd(lib, v=_tensor(sn=100)) == da.ERR_INVALID_ARG             # row stride < Dv
    assert _fwd(lib, q1=_tensor(sh=1028)) == da.ERR_INVALID_ARG           # stride not 16-byte multiple
    assert _fwd(lib, out=0x20004) == da.ERR_INVALID_ARG
    assert _fwd(lib, ind=7) == da.ERR_INVALID_ARG
    assert _fwd(lib, outd=7) == da.ERR_INVALID_ARG
    assert _fwd(lib, ind=da.F32, outd=da.F16, d=32, Dv=64) == da.ERR_INVALID_ARG  # fp32 inputs: f32/bf16 out
    assert _fwd(lib, lam=float("nan")) == da.ERR_INVALID_ARG
    assert _fwd(lib, eps=-1.0) == da.ERR_INVALID_ARG
    assert _fwd(lib, ws=None) == da.ERR_WORKSPACE
    assert _fwd(lib, wsb=8) == da.ERR_WORKSPACE
    assert _fwd(lib, ws=0x40010) == da.ERR_WORKSPACE                      # not 256-byte aligned
    assert _fwd(lib, d=32, Dv=64, q1=_tensor(sn=32), q2=_tensor(sn=32), k1=_tensor(sn=32),
                k2=_tensor(sn=32), v=_tensor(sn=64)) == da.ERR_UNSUPPORTED  # bf16 needs (64,128)/(128,256)
    assert _fwd(lib, ind=da.F16, d=32, Dv=64, q1=_tensor(sn=32), q2=_tensor(sn=32), k1=_tensor(sn=32),
                k2=_tensor(sn=32), v=_tensor(sn=64)) == da.ERR_UNSUPPORTED
    assert _fwd(lib, ind=da.F32, d=130, Dv=128, q1=_tensor(sn=132), q2=_tensor(sn=132), k1=_tensor(sn=132),
                k2=_tensor(sn=132)) == da.ERR_UNSUPPORTED


def test_decode_and_gemm_argument_validation(lib):
    t = _tensor()
    vp = ctypes.c_void_p
    call = lambda **kw: lib.diffattn_decode(
        vp(kw.get("q1", 0x1000)), vp(0x1000), kw.get("k1", t), t, kw.get("v", _tensor(sn=128)), None,
        kw.get("L", 64), vp(kw.get("out", 0x2000)), None, kw.get("B", 2), 2, kw.get("d", 64), 128, 0.5, 0.2, 1e-5,
        kw.get("S", 0), da.F32, vp(kw.get("ws", 0x4000)), kw.get("wsb", 256), None)
    assert call(B=0) == da.OK
    assert call(L=0) == da.ERR_INVALID_ARG
    assert call(q1=0) == da.ERR_INVALID_ARG
    assert call(S=300) == da.ERR_INVALID_ARG
    assert call(d=32, k1=_tensor(sn=32)) == da.ERR_UNSUPPORTED
    assert call(wsb=256) == da.ERR_WORKSPACE  # partial states need more than the control block
    n = ctypes.c_size_t()
    assert lib.diffattn_decode_workspace_size(64, 16, 8192, 64, 128, 4, ctypes.byref(n)) == da.OK
    assert n.value == 256 + 64 * 16 * 4 * 4 * 4 + 64 * 16 * 4 * 2 * 128 * 4
    for gemm in (lib.diffattn_gemm_bf16, lib.diffattn_gemm_f16):
        g = lambda **kw: gemm(vp(kw.get("A", 0x1000)), vp(0x2000), vp(0x3000), kw.get("M", 128), kw.get("N", 256),
                              64, kw.get("lda", 64), 256, 256, da.BF16, vp(0x4000), 256, None)
        assert g(M=0) == da.ERR_INVALID_ARG
        assert g(A=0x1008) == da.ERR_INVALID_ARG
        assert g(lda=60) == da.ERR_INVALID_ARG
        assert g(N=250) == da.ERR_INVALID_ARG


def test_noalloc_decode_argument_validation(lib):
    """The no-allocation decode checks its arguments like diffattn_decode before it
    looks up or writes its scratch, so these return without touching a device."""
    t = _tensor()
    vp = ctypes.c_void_p
    call = lambda **kw: lib.diffattn_decode_noalloc(
        vp(kw.get("q1", 0x1000)), vp(0x1000), kw.get("k1", t), t, kw.get("v", _tensor(sn=128)), None,
        kw.get("L", 64), vp(kw.get("out", 0x2000)), vp(kw.get("w")) if kw.get("w") else None, kw.get("B", 2), 2,
        kw.get("d", 64), 128, kw.get("lam", 0.5), 0.2, 1e-5, kw.get("S", 0), kw.get("outd", da.F32), None)
    assert call(B=0) == da.OK
    assert call(L=0) == da.ERR_INVALID_ARG
    assert call(S=300) == da.ERR_INVALID_ARG
    assert call(q1=0) == da.ERR_INVALID_ARG
    assert call(q1=0x1008) == da.ERR_INVALID_ARG                # misaligned
    assert call(out=0) == da.ERR_INVALID_ARG
    assert call(w=0x3004) == da.ERR_INVALID_ARG                 # misaligned norm weight
    assert call(k1=_tensor(sn=60)) == da.ERR_INVALID_ARG        # row stride < d
    assert call(outd=da.F16) == da.ERR_INVALID_ARG              # decode outputs fp32 or bf16
    assert call(lam=float("inf")) == da.ERR_INVALID_ARG
    assert call(d=32, k1=_tensor(sn=32)) == da.ERR_UNSUPPORTED
    assert lib.diffattn_decode_noalloc_read_error(None, None) == da.ERR_INVALID_ARG


@pytest.mark.parametrize("B,H,L,d", [(1, 1, 64, 64), (3, 4, 1000, 64), (64, 16, 8192, 64), (8, 16, 65536, 64),
                                     (2, 8, 300, 128), (128, 32, 4096, 128)])
def test_decode_auto_split_count_bounds(lib, B, H, L, d):
    """The automatic split count (read back from the workspace size) is at least 1, keeps at
    least 256 keys per split when it splits, and never exceeds 256."""
    Dv = 2 * d
    n = ctypes.c_size_t()
    assert lib.diffattn_decode_workspace_size(B, H, L, d, Dv, 0, ctypes.byref(n)) == da.OK
    per_split = B * H * (4 * 4 + 2 * Dv * 4)
    S, rem = divmod(n.value - 256, per_split)
    assert rem == 0 and 1 <= S <= 256
    assert S == 1 or L // S >= 256  # a split of a longer cache keeps at least 256 keys
    # an explicit count is taken as given (up to empty trailing splits)
    assert lib.diffattn_decode_workspace_size(B, H, L, d, Dv, 1, ctypes.byref(n)) == da.OK
    assert n.value == 256 + per_split


def test_paged_decode_argument_validation(lib):
    t = _tensor(sb=2 * 64 * 64, sh=64 * 64, sn=64)  # [pages, H_kv=2, 64, 64]
    vp = ctypes.c_void_p
    call = lambda **kw: lib.diffattn_decode_paged(
        vp(0x1000), vp(0x1000), t, t, _tensor(sb=2 * 64 * 128, sh=64 * 128, sn=128),
        None if kw.get("table", 1) is None else vp(0x3000), kw.get("max_pages", 4), 8,
        None if kw.get("lens", 1) is None else vp(0x3100), kw.get("L", 200), vp(0x2000), None, kw.get("B", 2),
        kw.get("H", 2), kw.get("g", 1), 64, 128, 0.5, 0.2, 1e-5, 0, da.F32, vp(0x4000), kw.get("wsb", 1 << 20), None)
    assert call(B=0) == da.OK
    assert call(g=0) == da.ERR_INVALID_ARG
    assert call(H=2, g=3) == da.ERR_INVALID_ARG        # kv_group must divide H
    assert call(L=300) == da.ERR_INVALID_ARG           # more than 64 * max_pages tokens
    assert call(table=None) == da.ERR_INVALID_ARG
    assert call(lens=None) == da.ERR_INVALID_ARG        # lengths are required with pages
    assert call(wsb=256) == da.ERR_WORKSPACE


def test_kv_append_argument_validation(lib):
    t = _tensor(sb=2 * 64 * 64, sh=64 * 64, sn=64)
    vp = ctypes.c_void_p
    call = lambda **kw: lib.diffattn_kv_append_paged(
        vp(kw.get("k1", 0x1000)), vp(0x1000), vp(0x1000), t, kw.get("k2", t), _tensor(sb=2 * 64 * 128, sh=64 * 128,
        sn=128), vp(0x3000), 4, 8, vp(0x3100), kw.get("B", 2), 2, kw.get("d", 64), 128, None)
    assert call(B=0) == da.OK
    assert call(k1=0) == da.ERR_INVALID_ARG
    assert call(k1=0x1004) == da.ERR_INVALID_ARG                 # not 16-byte aligned
    assert call(d=60) == da.ERR_INVALID_ARG                      # rows are copied in 16-byte chunks
    assert call(k2=_tensor(sb=4 * 64 * 64, sh=64 * 64, sn=64)) == da.ERR_INVALID_ARG  # K1/K2 strides differ


def test_fused_gemm_argument_validation(lib):
    """The layer's GEMMs with residual and SwiGLU epilogues reject bad arguments before any launch."""
    vp = ctypes.c_void_p
    res = lambda **kw: lib.diffattn_gemm_residual(
        vp(kw.get("A", 0x1000)), vp(0x2000), vp(kw.get("R", 0x3000)), vp(0x4000), vp(kw.get("C16", None)),
        vp(kw.get("gain", None)), None, kw.get("M", 128), kw.get("N", 256), 64, 64, 256, kw.get("ldr", 256), 256,
        kw.get("ldc16", 256), kw.get("ab", da.F16), kw.get("rd", da.F32), kw.get("c16d", da.F16), vp(0x8000),
        kw.get("wsb", 256), None)
    assert res(N=128) == da.ERR_INVALID_ARG          # N a multiple of 256
    assert res(ab=da.F32) == da.ERR_INVALID_ARG      # operands are 16-bit
    assert res(R=0) == da.ERR_INVALID_ARG
    assert res(R=0x3004) == da.ERR_INVALID_ARG       # 16-byte alignment
    assert res(ldr=200) == da.ERR_INVALID_ARG        # row stride below N
    assert res(gain=0x5000) == da.ERR_INVALID_ARG    # a gain without the copy
    assert res(C16=0x6000, c16d=da.F32) == da.ERR_INVALID_ARG
    assert res(C16=0x6000, ldc16=12) == da.ERR_INVALID_ARG
    assert res(M=0) == da.ERR_INVALID_ARG
    assert res(wsb=16) == da.ERR_WORKSPACE
    glu = lambda **kw: lib.diffattn_gemm_swiglu(
        vp(0x1000), vp(0x2000), vp(0x3000), vp(kw.get("sq", None)), kw.get("nsq", 8), kw.get("cnt", 512.0),
        kw.get("eps", 1e-5), 128, kw.get("F", 256), 64, 64, 512, 256, kw.get("ab", da.BF16), kw.get("hd", da.BF16),
        vp(0x8000), 256, None)
    assert glu(F=192) == da.ERR_INVALID_ARG          # F a multiple of 128
    assert glu(hd=da.F32) == da.ERR_INVALID_ARG      # H is 16-bit
    assert glu(sq=0x5000, nsq=0) == da.ERR_INVALID_ARG
    assert glu(sq=0x5000, cnt=0.0) == da.ERR_INVALID_ARG
    assert glu(sq=0x5000, eps=float("nan")) == da.ERR_INVALID_ARG


def test_host_prefill_argument_validation(lib):
    """diffattn_fwd_host rejects bad arguments before enqueuing anything; its buffer size is the
    workspace plus the device copies, each rounded up to 256 bytes."""
    vp = ctypes.c_void_p
    n = ctypes.c_size_t()
    assert lib.diffattn_fwd_host_buffer_size(2, 3, 100, 64, 128, da.BF16, da.BF16, ctypes.byref(n)) == da.OK
    r = lambda x: (x + 255) // 256 * 256
    assert n.value == 256 + 4 * r(2 * 3 * 100 * 64 * 2) + r(2 * 3 * 100 * 128 * 2) + r(2 * 100 * 3 * 128 * 2)
    assert lib.diffattn_fwd_host_buffer_size(2, 3, 100, 64, 128, 7, da.BF16, ctypes.byref(n)) == da.ERR_INVALID_ARG
    call = lambda **kw: lib.diffattn_fwd_host(
        vp(kw.get("q1", 0x1000)), vp(0x1000), vp(0x1000), vp(0x1000), vp(0x1000), vp(kw.get("out", 0x2000)), None,
        2, 3, 100, 64, 128, 1, 0.5, 0.2, 1e-5, da.BF16, da.BF16, kw.get("chunks", 0), vp(kw.get("buf", 0x100000)),
        kw.get("bytes", 1 << 24), None)
    assert call(q1=0) == da.ERR_INVALID_ARG
    assert call(out=0) == da.ERR_INVALID_ARG
    assert call(chunks=17) == da.ERR_INVALID_ARG
    assert call(chunks=-1) == da.ERR_INVALID_ARG
    assert call(bytes=1024) == da.ERR_WORKSPACE
    assert call(buf=0x100010) == da.ERR_WORKSPACE  # 256-byte alignment


def test_interleave_gate_up_layout():
    """Columns 256t..256t+127 of the interleaved weight are gate columns 128t.., the next 128 up's."""
    K, F = 4, 384
    wg = torch.arange(K * F, dtype=torch.float32).view(K, F)
    wu = -wg - 1
    w = da.interleave_gate_up(wg, wu)
    assert w.shape == (K, 2 * F)
    for t in range(F // 128):
        assert torch.equal(w[:, 256 * t: 256 * t + 128], wg[:, 128 * t: 128 * t + 128])
        assert torch.equal(w[:, 256 * t + 128: 256 * t + 256], wu[:, 128 * t: 128 * t + 128])
    with pytest.raises(ValueError):
        da.interleave_gate_up(wg[:, :100], wu[:, :100])


def test_layer_elementwise_argument_validation(lib):
    vp = ctypes.c_void_p
    norm = lambda **kw: lib.diffattn_add_rmsnorm(
        vp(kw.get("x", 0x1000)), kw.get("dt", da.BF16), None, vp(kw.get("y", 0x2000)), vp(0x3000),
        kw.get("nd", da.BF16), None, kw.get("M", 4), kw.get("N", 64), kw.get("eps", 1e-5), None)
    assert norm(M=0) == da.OK
    assert norm(x=0) == da.ERR_INVALID_ARG
    assert norm(x=0x1008) == da.ERR_INVALID_ARG                  # not 16-byte aligned
    assert norm(y=0x2004) == da.ERR_INVALID_ARG
    assert norm(N=60) == da.ERR_INVALID_ARG                      # rows move in 8-element chunks
    assert norm(dt=da.F16) == da.ERR_INVALID_ARG                 # x is bf16 or fp32
    assert norm(eps=-1.0) == da.ERR_INVALID_ARG
    assert norm(eps=float("nan")) == da.ERR_INVALID_ARG
    assert norm(M=-1) == da.ERR_INVALID_ARG
    assert norm(nd=da.F32) == da.ERR_INVALID_ARG                 # the normalised rows are bf16 or fp16
    glu = lambda **kw: lib.diffattn_swiglu(vp(kw.get("gu", 0x1000)), vp(kw.get("h", 0x2000)),
                                           kw.get("hd", da.F16), kw.get("M", 4), kw.get("H", 64), None)
    assert glu(M=0) == da.OK
    assert glu(gu=0) == da.ERR_INVALID_ARG
    assert glu(h=0x2002) == da.ERR_INVALID_ARG
    assert glu(H=12) == da.ERR_INVALID_ARG
    assert glu(M=-3) == da.ERR_INVALID_ARG
    assert glu(hd=da.F32) == da.ERR_INVALID_ARG


def _bwd(lib, **kw):
    a = dict(q1=_tensor(), q2=_tensor(), k1=_tensor(), k2=_tensor(), v=_tensor(sn=128), dy=0x20000, w=None,
             B=1, H=2, N=16, d=64, Dv=128, causal=1, lam=0.5, lam_init=0.2, eps=1e-5, ind=da.BF16,
             dq1=0x30000, dq2=0x30000, dk1=0x30000, dk2=0x30000, dv=0x30000, dlam=0x30000, dw=None,
             ws=0x40000, wsb=1 << 30, stream=None)
    a.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.diffattn_bwd(a["q1"], a["q2"], a["k1"], a["k2"], a["v"], vp(a["dy"]), vp(a["w"]), a["B"], a["H"],
                            a["N"], a["d"], a["Dv"], a["causal"], a["lam"], a["lam_init"], a["eps"], a["ind"],
                            vp(a["dq1"]), vp(a["dq2"]), vp(a["dk1"]), vp(a["dk2"]), vp(a["dv"]), vp(a["dlam"]),
                            vp(a["dw"]), vp(a["ws"]), a["wsb"], a["stream"])


def test_bwd_argument_validation(lib):
    assert _bwd(lib, B=0) == da.OK and _bwd(lib, N=0) == da.OK
    assert _bwd(lib, N=-1) == da.ERR_INVALID_ARG
    assert _bwd(lib, ind=7) == da.ERR_INVALID_ARG
    assert _bwd(lib, lam=float("inf")) == da.ERR_INVALID_ARG
    assert _bwd(lib, dy=None) == da.ERR_INVALID_ARG
    assert _bwd(lib, dk2=0x30004) == da.ERR_INVALID_ARG          # not 16-byte aligned
    assert _bwd(lib, dlam=None) == da.ERR_INVALID_ARG
    assert _bwd(lib, dw=0x30008) == da.ERR_INVALID_ARG
    assert _bwd(lib, v=_tensor(sn=100)) == da.ERR_INVALID_ARG
    assert _bwd(lib, d=48, q1=_tensor(sn=48), q2=_tensor(sn=48), k1=_tensor(sn=48),
                k2=_tensor(sn=48)) == da.ERR_UNSUPPORTED          # d a multiple of 32
    assert _bwd(lib, Dv=288, v=_tensor(sn=288)) == da.ERR_UNSUPPORTED
    n = ctypes.c_size_t()
    assert lib.diffattn_bwd_workspace_size(1, 2, 16, 64, 128, ctypes.byref(n)) == da.OK
    rows, parts = 2 * 16, 2 * 2
    r256 = lambda x: (x + 255) // 256 * 256
    assert n.value == 256 + r256(rows * 128 * 4) + r256(rows * 16) + r256(parts * 4) + r256(parts * 128 * 4)
    assert _bwd(lib, wsb=n.value - 1) == da.ERR_WORKSPACE
    assert _bwd(lib, ws=0x40010) == da.ERR_WORKSPACE


def test_training_pair_argument_validation(lib):
    """diffattn_fwd_train / diffattn_bwd_saved: the saved-state size and the checks that
    run before anything is launched."""
    n = ctypes.c_size_t()
    assert lib.diffattn_train_saved_size(1, 2, 16, 128, ctypes.byref(n)) == da.OK
    rows = 2 * 16
    r256 = lambda x: (x + 255) // 256 * 256
    assert n.value == r256(rows * 128 * 4) + r256(rows * 128 * 2) + r256(rows * 8)  # x, O2/l2, L1 and L2
    for B, H, N in ((1, 1, 1), (3, 5, 130), (4, 16, 2048), (2, 3, 16383)):
        assert lib.diffattn_train_saved_size(B, H, N, 128, ctypes.byref(n)) == da.OK
        r = B * H * N
        assert n.value == r256(r * 128 * 4) + r256(r * 128 * 2) + r256(r * 8), (B, H, N)
    assert lib.diffattn_train_saved_size(1, 2, 16, 128, ctypes.byref(n)) == da.OK
    assert lib.diffattn_train_saved_size(1, -2, 16, 128, ctypes.byref(n)) == da.ERR_INVALID_ARG
    assert lib.diffattn_train_saved_size(1, 2, 16, 128, None) == da.ERR_INVALID_ARG
    nbytes = n.value

    def train(**kw):
        a = dict(q1=_tensor(), q2=_tensor(), k1=_tensor(), k2=_tensor(), v=_tensor(sn=128), out=0x20000, w=None,
                 B=1, H=2, N=16, d=64, Dv=128, causal=1, lam=0.5, lam_init=0.2, eps=1e-5, ind=da.BF16, outd=da.BF16,
                 saved=0x50000, savedb=nbytes, ws=0x40000, wsb=256, stream=None)
        a.update(kw)
        vp = lambda x: None if x is None else ctypes.c_void_p(x)
        return lib.diffattn_fwd_train(a["q1"], a["q2"], a["k1"], a["k2"], a["v"], vp(a["out"]), vp(a["w"]), a["B"],
                                      a["H"], a["N"], a["d"], a["Dv"], a["causal"], a["lam"], a["lam_init"], a["eps"],
                                      a["ind"], a["outd"], vp(a["saved"]), a["savedb"], vp(a["ws"]), a["wsb"],
                                      a["stream"])

    def bwd(**kw):
        a = dict(q1=_tensor(), q2=_tensor(), k1=_tensor(), k2=_tensor(), v=_tensor(sn=128), dy=0x20000, w=None,
                 B=1, H=2, N=16, d=64, Dv=128, causal=1, lam=0.5, lam_init=0.2, eps=1e-5, ind=da.BF16,
                 saved=0x50000, savedb=nbytes, dq1=0x30000, dq2=0x30000, dk1=0x30000, dk2=0x30000, dv=0x30000,
                 dlam=0x30000, dw=None, ws=0x40000, wsb=1 << 30, stream=None)
        a.update(kw)
        vp = lambda x: None if x is None else ctypes.c_void_p(x)
        return lib.diffattn_bwd_saved(a["q1"], a["q2"], a["k1"], a["k2"], a["v"], vp(a["dy"]), vp(a["w"]), a["B"],
                                      a["H"], a["N"], a["d"], a["Dv"], a["causal"], a["lam"], a["lam_init"], a["eps"],
                                      a["ind"], vp(a["saved"]), a["savedb"], vp(a["dq1"]), vp(a["dq2"]), vp(a["dk1"]),
                                      vp(a["dk2"]), vp(a["dv"]), vp(a["dlam"]), vp(a["dw"]), vp(a["ws"]), a["wsb"],
                                      a["stream"])

    for call in (train, bwd):
        assert call(B=0) == da.OK and call(N=0) == da.OK                    # nothing to do
        assert call(ind=da.F32) == da.ERR_UNSUPPORTED                       # tensor-core path only
        assert call(d=128, q1=_tensor(sn=128), q2=_tensor(sn=128), k1=_tensor(sn=128),
                    k2=_tensor(sn=128), Dv=256, v=_tensor(sn=256)) == da.ERR_UNSUPPORTED
        assert call(saved=None) == da.ERR_INVALID_ARG
        assert call(saved=0x50010) == da.ERR_INVALID_ARG                    # not 256-byte aligned
        assert call(savedb=nbytes - 1) == da.ERR_INVALID_ARG
        assert call(lam=float("nan")) == da.ERR_INVALID_ARG
    assert train(out=0x20004) == da.ERR_INVALID_ARG
    assert bwd(dy=None) == da.ERR_INVALID_ARG


def test_host_lambda_backward_matches_oracle(lib):
    r = np.random.default_rng(3)
    vecs = [(0.2 * r.standard_normal(64)).astype(np.float32) for _ in range(4)]
    got = da.diffattn_lambda_bwd(*vecs, -1.7)
    ref = orc.reparam_lambda_bwd(*vecs, -1.7)
    for g, e in zip(got, ref):
        np.testing.assert_allclose(g.numpy(), e, rtol=1e-6, atol=1e-9)
    with pytest.raises(da.DiffAttnError):
        da.diffattn_lambda_bwd(*vecs, float("nan"))


def test_fp8_cache_argument_validation(lib):
    t8 = _tensor(sb=2 * 64 * 64, sh=64 * 64, sn=64)      # [pages, 2, 64, 64] bytes
    v8 = _tensor(sb=2 * 64 * 128, sh=64 * 128, sn=128)
    vp = ctypes.c_void_p
    dec = lambda **kw: lib.diffattn_decode_paged_fp8(
        vp(0x1000), vp(0x1000), kw.get("k", t8), t8, v8, vp(0x3000), 4, 8, vp(0x3100), 200, vp(0x2000), None,
        kw.get("B", 2), 2, 1, 64, 128, 0.5, 0.2, 1e-5, kw.get("ks", 0.01), 0.01, kw.get("vs", 0.01), 0, da.F32,
        vp(0x4000), 1 << 20, None)
    assert dec(B=0) == da.OK
    assert dec(ks=0.0) == da.ERR_INVALID_ARG
    assert dec(vs=float("inf")) == da.ERR_INVALID_ARG
    assert dec(ks=-1.0) == da.ERR_INVALID_ARG
    assert dec(k=_tensor(sb=2 * 64 * 64, sh=64 * 64, sn=72)) == da.ERR_INVALID_ARG  # 72-byte rows: not 16-multiple
    app = lambda **kw: lib.diffattn_kv_append_paged_fp8(
        vp(0x1000), vp(0x1000), vp(0x1000), t8, t8, v8, vp(0x3000), 4, 8, vp(0x3100), kw.get("B", 2), 2, 64, 128,
        kw.get("ks", 0.01), 0.01, 0.01, None)
    assert app(B=0) == da.OK
    assert app(ks=float("nan")) == da.ERR_INVALID_ARG


def test_python_wrappers_reject_inconsistent_arguments(lib):
    """Checks the bindings make before any device work (CPU tensors suffice)."""
    t = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16)
    v = torch.zeros(1, 2, 64, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        da.diffattn_bwd(t, t, t, t, v, torch.zeros(1, 64, 2, 128, dtype=torch.bfloat16), 0.5, 0.2)
    p8 = torch.zeros(4, 2, 64, 64, dtype=torch.float8_e4m3fn)
    v8 = torch.zeros(4, 2, 64, 128, dtype=torch.float8_e4m3fn)
    pb = torch.zeros(4, 2, 64, 64, dtype=torch.bfloat16)
    q = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    table, lens = torch.zeros(1, 4, dtype=torch.int32), torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="scales"):
        da.diffattn_decode_paged(q, q, p8, p8, v8, table, lens, 0.5, 0.2, L=64)             # fp8 without scales
    with pytest.raises(ValueError, match="scales"):
        da.diffattn_decode_paged(q, q, pb, pb, pb, table, lens, 0.5, 0.2, L=64, scales=(1, 1, 1))
    with pytest.raises(ValueError, match="scales"):
        da.diffattn_decode_paged(q, q, p8, pb, v8, table, lens, 0.5, 0.2, L=64, scales=(1, 1, 1))
    with pytest.raises(ValueError, match="scales"):
        da.diffattn_kv_append_paged(q, q, torch.zeros(1, 2, 128, dtype=torch.bfloat16), p8, p8, v8, table, lens)
    with pytest.raises(ValueError, match="both"):
        da.gemm(torch.zeros(8, 8, dtype=torch.bfloat16), torch.zeros(8, 8, dtype=torch.float16))


def test_python_binding_refuses_without_library(tmp_path):
    saved = da._lib
    da._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            da.load_library(str(tmp_path / "nope.so"))
    finally:
        da._lib = saved

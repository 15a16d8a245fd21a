"""Python binding of libdiffattn.so (causal multi-head differential attention, GB300).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels. PyTorch supplies device memory and the current CUDA stream. The
library must have been built (``differential_attention_02_gb300.build.build()``);
if it is missing, every call raises instead of computing anything elsewhere.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# DIFFATTN_LIBRARY selects another build of the library, e.g. libdiffattn_debug.so.
LIB_PATH = os.environ.get("DIFFATTN_LIBRARY") or os.path.join(_PKG, "libdiffattn.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(6)
F32, BF16, F16 = 0, 1, 2

EXPORTED = ("diffattn_status_string", "diffattn_lambda", "diffattn_fwd", "diffattn_fwd_workspace_size",
            "diffattn_decode", "diffattn_decode_workspace_size", "diffattn_gemm_bf16", "diffattn_gemm_f16",
            "diffattn_gemm_workspace_size", "diffattn_read_error", "diffattn_decode_noalloc",
            "diffattn_decode_paged", "diffattn_kv_append_paged", "diffattn_add_rmsnorm", "diffattn_swiglu",
            "diffattn_bwd", "diffattn_bwd_workspace_size", "diffattn_lambda_bwd", "diffattn_decode_paged_fp8",
            "diffattn_kv_append_paged_fp8", "diffattn_decode_noalloc_read_error",
            "diffattn_selftest_timeout", "diffattn_gemm_residual", "diffattn_gemm_swiglu", "diffattn_fwd_host",
            "diffattn_fwd_host_buffer_size", "diffattn_train_saved_size", "diffattn_fwd_train",
            "diffattn_bwd_saved")


class DiffAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Tensor4(ctypes.Structure):
    """diffattn_tensor: pointer plus (b, h, n) strides in elements."""
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64),
                ("stride_n", ctypes.c_int64)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libdiffattn.so and declares its signatures (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with differential_attention_02_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    fp = ctypes.POINTER(ctypes.c_float)
    lib.diffattn_status_string.restype = ctypes.c_char_p
    lib.diffattn_status_string.argtypes = [i32]
    lib.diffattn_lambda.restype = i32
    lib.diffattn_lambda.argtypes = [fp, fp, fp, fp, i32, i32, f32, fp, fp]
    lib.diffattn_fwd.restype = i32
    lib.diffattn_fwd.argtypes = [Tensor4] * 5 + [vp, vp, i32, i32, i32, i32, i32, i32, f32, f32, f32, i32, i32,
                                                 vp, sz, vp]
    lib.diffattn_fwd_workspace_size.restype = i32
    lib.diffattn_fwd_workspace_size.argtypes = [i32] * 5 + [ctypes.POINTER(sz)]
    lib.diffattn_decode.restype = i32
    lib.diffattn_decode.argtypes = [vp, vp, Tensor4, Tensor4, Tensor4, vp, i32, vp, vp, i32, i32, i32, i32, f32,
                                    f32, f32, i32, i32, vp, sz, vp]
    lib.diffattn_decode_workspace_size.restype = i32
    lib.diffattn_decode_workspace_size.argtypes = [i32] * 6 + [ctypes.POINTER(sz)]
    lib.diffattn_gemm_bf16.restype = i32
    lib.diffattn_gemm_bf16.argtypes = [vp, vp, vp, i32, i32, i32, i64, i64, i64, i32, vp, sz, vp]
    lib.diffattn_gemm_f16.restype = i32
    lib.diffattn_gemm_f16.argtypes = lib.diffattn_gemm_bf16.argtypes
    lib.diffattn_gemm_residual.restype = i32
    lib.diffattn_gemm_residual.argtypes = [vp] * 7 + [i32] * 3 + [i64] * 5 + [i32] * 3 + [vp, sz, vp]
    lib.diffattn_gemm_swiglu.restype = i32
    lib.diffattn_gemm_swiglu.argtypes = [vp, vp, vp, vp, i32, f32, f32, i32, i32, i32, i64, i64, i64, i32, i32, vp, sz,
                                         vp]
    lib.diffattn_fwd_host.restype = i32
    lib.diffattn_fwd_host.argtypes = [vp] * 7 + [i32] * 6 + [f32] * 3 + [i32] * 3 + [vp, sz, vp]
    lib.diffattn_fwd_host_buffer_size.restype = i32
    lib.diffattn_fwd_host_buffer_size.argtypes = [i32] * 7 + [ctypes.POINTER(sz)]
    lib.diffattn_gemm_workspace_size.restype = i32
    lib.diffattn_gemm_workspace_size.argtypes = [i32, i32, i32, ctypes.POINTER(sz)]
    lib.diffattn_decode_noalloc.restype = i32
    lib.diffattn_decode_noalloc.argtypes = [vp, vp, Tensor4, Tensor4, Tensor4, vp, i32, vp, vp, i32, i32, i32, i32,
                                            f32, f32, f32, i32, i32, vp]
    lib.diffattn_decode_noalloc_read_error.restype = i32
    lib.diffattn_decode_noalloc_read_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.diffattn_decode_paged.restype = i32
    lib.diffattn_decode_paged.argtypes = [vp, vp, Tensor4, Tensor4, Tensor4, vp, i32, i32, vp, i32, vp, vp, i32, i32,
                                          i32, i32, i32, f32, f32, f32, i32, i32, vp, sz, vp]
    lib.diffattn_kv_append_paged.restype = i32
    lib.diffattn_kv_append_paged.argtypes = [vp, vp, vp, Tensor4, Tensor4, Tensor4, vp, i32, i32, vp, i32, i32, i32,
                                             i32, vp]
    lib.diffattn_decode_paged_fp8.restype = i32
    lib.diffattn_decode_paged_fp8.argtypes = [vp, vp, Tensor4, Tensor4, Tensor4, vp, i32, i32, vp, i32, vp, vp, i32,
                                              i32, i32, i32, i32, f32, f32, f32, f32, f32, f32, i32, i32, vp, sz, vp]
    lib.diffattn_kv_append_paged_fp8.restype = i32
    lib.diffattn_kv_append_paged_fp8.argtypes = [vp, vp, vp, Tensor4, Tensor4, Tensor4, vp, i32, i32, vp, i32, i32,
                                                 i32, i32, f32, f32, f32, vp]
    lib.diffattn_add_rmsnorm.restype = i32
    lib.diffattn_add_rmsnorm.argtypes = [vp, i32, vp, vp, vp, i32, vp, i32, i32, f32, vp]
    lib.diffattn_swiglu.restype = i32
    lib.diffattn_swiglu.argtypes = [vp, vp, i32, i32, i32, vp]
    lib.diffattn_bwd.restype = i32
    lib.diffattn_bwd.argtypes = [Tensor4] * 5 + [vp, vp] + [i32] * 6 + [f32] * 3 + [i32] + [vp] * 7 + [vp, sz, vp]
    lib.diffattn_bwd_workspace_size.restype = i32
    lib.diffattn_bwd_workspace_size.argtypes = [i32] * 5 + [ctypes.POINTER(sz)]
    lib.diffattn_train_saved_size.restype = i32
    lib.diffattn_train_saved_size.argtypes = [i32] * 4 + [ctypes.POINTER(sz)]
    lib.diffattn_fwd_train.restype = i32
    lib.diffattn_fwd_train.argtypes = [Tensor4] * 5 + [vp, vp] + [i32] * 6 + [f32] * 3 + [i32, i32, vp, sz, vp, sz, vp]
    lib.diffattn_bwd_saved.restype = i32
    lib.diffattn_bwd_saved.argtypes = ([Tensor4] * 5 + [vp, vp] + [i32] * 6 + [f32] * 3 + [i32, vp, sz] + [vp] * 7 +
                                       [vp, sz, vp])
    fpp = ctypes.POINTER(ctypes.c_float)
    lib.diffattn_lambda_bwd.restype = i32
    lib.diffattn_lambda_bwd.argtypes = [fpp] * 4 + [i32, f32] + [fpp] * 4
    lib.diffattn_selftest_timeout.restype = i32
    lib.diffattn_selftest_timeout.argtypes = [vp, sz, vp]
    lib.diffattn_read_error.restype = i32
    lib.diffattn_read_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().diffattn_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != OK:
        raise DiffAttnError(status, what)


def _stream_ptr(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt) -> int:
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float16:
        return F16
    raise ValueError(f"unsupported dtype {dt}")


def _t4(t: torch.Tensor) -> Tensor4:
    """[B, H, rows, width] view with a contiguous last dim -> diffattn_tensor."""
    if t.dim() != 4 or t.stride(-1) != 1:
        raise ValueError("operand must be 4-D [B, H, rows, width] with a contiguous last dimension")
    return Tensor4(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))


# ------------------------------------------------------------------ workspace
_ws_cache: dict = {}


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-initialised, 256-byte-aligned device buffer of at least nbytes (cached per device)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    key = dev.index
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(int(nbytes), 256) + 256, dtype=torch.uint8, device=dev)
        _ws_cache[key] = buf
    off = (-buf.data_ptr()) % 256
    return buf[off:]


def read_error(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error word of a workspace."""
    code = ctypes.c_int32(0)
    st = load_library().diffattn_read_error(ctypes.c_void_p(ws.data_ptr()), _stream_ptr(stream), ctypes.byref(code))
    if st not in (OK, ERR_TIMEOUT):
        _check(st, "diffattn_read_error")
    return code.value


# ------------------------------------------------------------------ entry points
def diffattn_lambda(lq1, lk1, lq2, lk2, layer: int, lambda_init_override: float | None = None):
    """lambda and lambda_init (host computation in double, returned as floats)."""
    vs = [torch.as_tensor(v, dtype=torch.float32).contiguous().reshape(-1) for v in (lq1, lk1, lq2, lk2)]
    d = vs[0].numel()
    if any(v.numel() != d for v in vs):
        raise ValueError("lambda vectors must have one common length")
    lam, lam_init = ctypes.c_float(), ctypes.c_float()
    fp = ctypes.POINTER(ctypes.c_float)
    ptrs = [ctypes.cast(v.data_ptr(), fp) for v in vs]
    ov = -1.0 if lambda_init_override is None else float(lambda_init_override)
    _check(load_library().diffattn_lambda(*ptrs, d, int(layer), ov, ctypes.byref(lam), ctypes.byref(lam_init)),
           "diffattn_lambda")
    return lam.value, lam_init.value


def diffattn_fwd(q1, q2, k1, k2, v, lam: float, lam_init: float, eps: float = 1e-5, norm_weight=None,
                 causal: bool = True, out_dtype=torch.float32, out=None, ws=None, stream=None) -> torch.Tensor:
    """Fused prefill. q1,q2,k1,k2: [B,H,N,d]; v: [B,H,N,Dv] (CUDA, fp32, bf16 or fp16). Returns [B,N,H,Dv]."""
    B, H, N, d = q1.shape
    Dv = v.shape[-1]
    for t in (q1, q2, k1, k2, v):
        if not t.is_cuda or t.dtype != q1.dtype:
            raise ValueError("all operands must be CUDA tensors of one dtype")
    if out is None:
        out = torch.empty((B, N, H, Dv), dtype=out_dtype, device=q1.device)
    lib = load_library()
    if ws is None:
        nbytes = ctypes.c_size_t()
        _check(lib.diffattn_fwd_workspace_size(B, H, N, d, Dv, ctypes.byref(nbytes)), "diffattn_fwd_workspace_size")
        ws = workspace(nbytes.value, q1.device)
    w = None if norm_weight is None else ctypes.c_void_p(norm_weight.data_ptr())
    _check(lib.diffattn_fwd(_t4(q1), _t4(q2), _t4(k1), _t4(k2), _t4(v), ctypes.c_void_p(out.data_ptr()), w,
                            B, H, N, d, Dv, int(bool(causal)), float(lam), float(lam_init), float(eps),
                            _dtype_code(q1.dtype), _dtype_code(out.dtype), ctypes.c_void_p(ws.data_ptr()),
                            ws.numel(), _stream_ptr(stream)), "diffattn_fwd")
    return out


def train_saved_bytes(B, H, N, Dv) -> int:
    n = ctypes.c_size_t()
    _check(load_library().diffattn_train_saved_size(B, H, N, Dv, ctypes.byref(n)), "diffattn_train_saved_size")
    return n.value


def saved_state(B, H, N, Dv, device=None) -> torch.Tensor:
    """A buffer of its own (not the cached workspace: the state must outlive other calls)
    for diffattn_fwd_train's saved state: 256-byte aligned, train_saved_bytes() long."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    n = train_saved_bytes(B, H, N, Dv)
    buf = torch.empty(n + 256, dtype=torch.uint8, device=dev)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + n]


def diffattn_fwd_train(q1, q2, k1, k2, v, lam: float, lam_init: float, eps: float = 1e-5, norm_weight=None,
                       causal: bool = True, out_dtype=torch.float32, out=None, saved=None, ws=None, stream=None):
    """diffattn_fwd that also saves the state diffattn_bwd(..., saved=...) starts from (bf16/fp16,
    d=64, Dv=128). Returns (out, saved); `saved` is a uint8 device buffer of train_saved_bytes()."""
    B, H, N, d = q1.shape
    Dv = v.shape[-1]
    for t in (q1, q2, k1, k2, v):
        if not t.is_cuda or t.dtype != q1.dtype:
            raise ValueError("all operands must be CUDA tensors of one dtype")
    dev = q1.device
    if out is None:
        out = torch.empty((B, N, H, Dv), dtype=out_dtype, device=dev)
    if saved is None:
        saved = saved_state(B, H, N, Dv, dev)
    lib = load_library()
    if ws is None:
        ws = workspace(256, dev)
    w = None if norm_weight is None else ctypes.c_void_p(norm_weight.data_ptr())
    _check(lib.diffattn_fwd_train(_t4(q1), _t4(q2), _t4(k1), _t4(k2), _t4(v), ctypes.c_void_p(out.data_ptr()), w,
                                  B, H, N, d, Dv, int(bool(causal)), float(lam), float(lam_init), float(eps),
                                  _dtype_code(q1.dtype), _dtype_code(out.dtype), ctypes.c_void_p(saved.data_ptr()),
                                  saved.numel(), ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_ptr(stream)),
           "diffattn_fwd_train")
    return out, saved


def diffattn_bwd(q1, q2, k1, k2, v, dy, lam: float, lam_init: float, eps: float = 1e-5, norm_weight=None,
                 causal: bool = True, want_dnorm_weight: bool = False, ws=None, stream=None, saved=None) -> dict:
    """Backward of diffattn_fwd. Operands as for diffattn_fwd (one dtype: fp32, bf16 or fp16); dy
    [B,N,H,Dv] of that dtype. Returns dq1, dq2, dk1, dk2 [B,H,N,d] fp32, dv [B,H,N,Dv] fp32, dlam
    (a 1-element fp32 device tensor) and dw ([Dv] fp32, or None). With `saved` (from
    diffattn_fwd_train on the same inputs) it starts from that state (diffattn_bwd_saved)."""
    B, H, N, d = q1.shape
    Dv = v.shape[-1]
    for t in (q1, q2, k1, k2, v, dy):
        if not t.is_cuda or t.dtype != q1.dtype:
            raise ValueError("all operands and dy must be CUDA tensors of one dtype")
    if tuple(dy.shape) != (B, N, H, Dv) or not dy.is_contiguous():
        raise ValueError("dy must be a contiguous [B, N, H, Dv] tensor")
    lib = load_library()
    dev = q1.device
    g = {k: torch.empty((B, H, N, Dv if k == "dv" else d), dtype=torch.float32, device=dev)
         for k in ("dq1", "dq2", "dk1", "dk2", "dv")}
    g["dlam"] = torch.empty(4, dtype=torch.float32, device=dev)[:1]
    g["dw"] = torch.empty(Dv, dtype=torch.float32, device=dev) if want_dnorm_weight else None
    if ws is None:
        nbytes = ctypes.c_size_t()
        _check(lib.diffattn_bwd_workspace_size(B, H, N, d, Dv, ctypes.byref(nbytes)), "diffattn_bwd_workspace_size")
        ws = workspace(nbytes.value, dev)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    head = (_t4(q1), _t4(q2), _t4(k1), _t4(k2), _t4(v), ptr(dy), ptr(norm_weight), B, H, N, d, Dv,
            int(bool(causal)), float(lam), float(lam_init), float(eps), _dtype_code(q1.dtype))
    grads = (ptr(g["dq1"]), ptr(g["dq2"]), ptr(g["dk1"]), ptr(g["dk2"]), ptr(g["dv"]), ptr(g["dlam"]), ptr(g["dw"]))
    tail = (ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_ptr(stream))
    if saved is None:
        _check(lib.diffattn_bwd(*head, *grads, *tail), "diffattn_bwd")
    else:
        _check(lib.diffattn_bwd_saved(*head, ptr(saved), saved.numel(), *grads, *tail), "diffattn_bwd_saved")
    return g


def bwd_workspace_bytes(B, H, N, d, Dv) -> int:
    n = ctypes.c_size_t()
    _check(load_library().diffattn_bwd_workspace_size(B, H, N, d, Dv, ctypes.byref(n)), "diffattn_bwd_workspace_size")
    return n.value


def diffattn_lambda_bwd(lq1, lk1, lq2, lk2, dlam: float):
    """Gradients of lambda with respect to the four lambda vectors (host, double), given dlam."""
    vs = [torch.as_tensor(v, dtype=torch.float32).contiguous().reshape(-1) for v in (lq1, lk1, lq2, lk2)]
    d = vs[0].numel()
    if any(v.numel() != d for v in vs):
        raise ValueError("lambda vectors must have one common length")
    outs = [torch.empty(d, dtype=torch.float32) for _ in range(4)]
    fp = ctypes.POINTER(ctypes.c_float)
    c = lambda t: ctypes.cast(t.data_ptr(), fp)
    _check(load_library().diffattn_lambda_bwd(*(c(v) for v in vs), d, float(dlam), *(c(o) for o in outs)),
           "diffattn_lambda_bwd")
    return tuple(outs)


def decode_workspace_bytes(B, H, L, d, Dv, num_splits=0) -> int:
    n = ctypes.c_size_t()
    _check(load_library().diffattn_decode_workspace_size(B, H, L, d, Dv, num_splits, ctypes.byref(n)),
           "diffattn_decode_workspace_size")
    return n.value


def diffattn_decode(q1, q2, k1_cache, k2_cache, v_cache, lam: float, lam_init: float, seq_lens=None, L=None,
                    eps: float = 1e-5, norm_weight=None, num_splits: int = 0, out_dtype=torch.float32, out=None,
                    ws=None, stream=None) -> torch.Tensor:
    """Split-KV decode. q: [B,H,d]; caches [B,H,Lmax,*] bf16; seq_lens int32 [B] (CUDA) or None. -> [B,H,Dv]."""
    B, H, d = q1.shape
    Dv = v_cache.shape[-1]
    L = k1_cache.shape[2] if L is None else int(L)
    if out is None:
        out = torch.empty((B, H, Dv), dtype=out_dtype, device=q1.device)
    nbytes = decode_workspace_bytes(B, H, L, d, Dv, num_splits)
    ws = workspace(nbytes, q1.device) if ws is None else ws
    sl = None
    if seq_lens is not None:
        if seq_lens.dtype != torch.int32 or not seq_lens.is_cuda:
            raise ValueError("seq_lens must be a CUDA int32 tensor")
        sl = ctypes.c_void_p(seq_lens.data_ptr())
    w = None if norm_weight is None else ctypes.c_void_p(norm_weight.data_ptr())
    _check(load_library().diffattn_decode(
        ctypes.c_void_p(q1.data_ptr()), ctypes.c_void_p(q2.data_ptr()), _t4(k1_cache), _t4(k2_cache), _t4(v_cache),
        sl, L, ctypes.c_void_p(out.data_ptr()), w, B, H, d, Dv, float(lam), float(lam_init), float(eps),
        int(num_splits), _dtype_code(out.dtype), ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_ptr(stream)),
        "diffattn_decode")
    return out


def _is_fp8(t) -> bool:
    return t.dtype in (torch.float8_e4m3fn, torch.uint8)


def diffattn_decode_paged(q1, q2, k1_pages, k2_pages, v_pages, block_table, seq_lens, lam: float, lam_init: float,
                          L: int, kv_group: int = 1, eps: float = 1e-5, norm_weight=None, num_splits: int = 0,
                          out_dtype=torch.float32, out=None, ws=None, stream=None, scales=None) -> torch.Tensor:
    """Split-KV decode against a paged KV cache. q: [B,H,d]; pages [num_pages, H/kv_group, 64, *] bf16, or
    fp8 e4m3 (torch.float8_e4m3fn or uint8 bytes) with scales = (k1_scale, k2_scale, v_scale); block_table
    int32 [B, max_pages] and seq_lens int32 [B] on the GPU; L = the largest length. -> [B,H,Dv]."""
    fp8 = _is_fp8(k1_pages)
    if fp8 != (scales is not None) or any(_is_fp8(t) != fp8 for t in (k2_pages, v_pages)):
        raise ValueError("fp8 pages (all three) go with scales, bf16 pages without")
    B, H, d = q1.shape
    Dv = v_pages.shape[-1]
    num_pages, max_pages = k1_pages.shape[0], block_table.shape[1]
    for t in (block_table, seq_lens):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("block_table and seq_lens must be contiguous CUDA int32 tensors")
    if out is None:
        out = torch.empty((B, H, Dv), dtype=out_dtype, device=q1.device)
    nbytes = decode_workspace_bytes(B, H, int(L), d, Dv, num_splits)
    ws = workspace(nbytes, q1.device) if ws is None else ws
    w = None if norm_weight is None else ctypes.c_void_p(norm_weight.data_ptr())
    lib = load_library()
    head = (ctypes.c_void_p(q1.data_ptr()), ctypes.c_void_p(q2.data_ptr()), _t4(k1_pages), _t4(k2_pages),
            _t4(v_pages), ctypes.c_void_p(block_table.data_ptr()), max_pages, num_pages,
            ctypes.c_void_p(seq_lens.data_ptr()), int(L), ctypes.c_void_p(out.data_ptr()), w, B, H, int(kv_group), d,
            Dv, float(lam), float(lam_init), float(eps))
    tail = (int(num_splits), _dtype_code(out.dtype), ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_ptr(stream))
    if fp8:
        _check(lib.diffattn_decode_paged_fp8(*head, *(float(x) for x in scales), *tail), "diffattn_decode_paged_fp8")
    else:
        _check(lib.diffattn_decode_paged(*head, *tail), "diffattn_decode_paged")
    return out


def diffattn_kv_append_paged(k1_new, k2_new, v_new, k1_pages, k2_pages, v_pages, block_table, seq_lens,
                             stream=None, scales=None) -> None:
    """Writes the new token's K1, K2, V rows ([B, H_kv, *] bf16) into the paged cache at position
    seq_lens[b] - 1 of each sequence (pages [num_pages, H_kv, 64, *], block_table [B, max_pages]).
    fp8 pages take scales = (k1_scale, k2_scale, v_scale) and store e4m3(x / scale)."""
    B, Hk, d = k1_new.shape
    Dv = v_new.shape[-1]
    for t in (k1_new, k2_new, v_new):
        if not t.is_contiguous():
            raise ValueError("new-token rows must be contiguous")
    fp8 = _is_fp8(k1_pages)
    if fp8 != (scales is not None) or any(_is_fp8(t) != fp8 for t in (k2_pages, v_pages)):
        raise ValueError("fp8 pages (all three) go with scales, bf16 pages without")
    args = (ctypes.c_void_p(k1_new.data_ptr()), ctypes.c_void_p(k2_new.data_ptr()), ctypes.c_void_p(v_new.data_ptr()),
            _t4(k1_pages), _t4(k2_pages), _t4(v_pages), ctypes.c_void_p(block_table.data_ptr()), block_table.shape[1],
            k1_pages.shape[0], ctypes.c_void_p(seq_lens.data_ptr()), B, Hk, d, Dv)
    lib = load_library()
    if fp8:
        _check(lib.diffattn_kv_append_paged_fp8(*args, *(float(x) for x in scales), _stream_ptr(stream)),
               "diffattn_kv_append_paged_fp8")
    else:
        _check(lib.diffattn_kv_append_paged(*args, _stream_ptr(stream)), "diffattn_kv_append_paged")


def add_rmsnorm(x, z=None, weight=None, eps: float = 1e-5, want_y: bool = False, want_n: bool = True,
                n_dtype=torch.bfloat16, stream=None):
    """Row-wise y = x + z and n = RMSNorm(y) * weight over the last dimension.
    x [.., N] bf16 or fp32, z fp32 or None. Returns (y fp32 or None, n of n_dtype
    (bf16 or fp16) or None)."""
    N = x.shape[-1]
    M = x.numel() // N
    y = torch.empty(x.shape, dtype=torch.float32, device=x.device) if want_y else None
    n = torch.empty(x.shape, dtype=n_dtype, device=x.device) if want_n else None
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    _check(load_library().diffattn_add_rmsnorm(
        ptr(x), F32 if x.dtype == torch.float32 else BF16, ptr(z), ptr(y), ptr(n), _dtype_code(n_dtype), ptr(weight),
        M, N, float(eps), _stream_ptr(stream)), "diffattn_add_rmsnorm")
    return y, n


def swiglu(gate_up, out_dtype=torch.bfloat16, stream=None):
    """h = SiLU(g) * u for rows [g | u] of gate_up ([M, 2H] fp16). Returns [M, H] of out_dtype."""
    M, H2 = gate_up.shape
    h = torch.empty((M, H2 // 2), dtype=out_dtype, device=gate_up.device)
    _check(load_library().diffattn_swiglu(ctypes.c_void_p(gate_up.data_ptr()), ctypes.c_void_p(h.data_ptr()),
                                          _dtype_code(out_dtype), M, H2 // 2, _stream_ptr(stream)),
           "diffattn_swiglu")
    return h


def interleave_gate_up(w_gate, w_up):
    """[K, F] gate and up weights -> [K, 2F] with 128-column blocks interleaved: columns
    256 t .. 256 t + 127 hold w_gate[:, 128 t : 128 t + 128], the next 128 w_up's (the layout
    gemm_swiglu reads). F a multiple of 128. A one-time weight transform."""
    K, F = w_gate.shape
    if w_up.shape != (K, F) or F % 128:
        raise ValueError("w_gate and w_up [K, F] with F a multiple of 128")
    return torch.stack([w_gate.reshape(K, F // 128, 128), w_up.reshape(K, F // 128, 128)], dim=2).reshape(
        K, 2 * F).contiguous()


def layer_fwd(x, w_q, w_k, w_v, w_o, w_gu, w_down, n_heads: int, lam: float, lam_init: float,
              eps: float = 1e-5, norm1_weight=None, norm2_weight=None, head_weight=None, ws=None, stream=None,
              w_qkv=None):
    """One DIFF Transformer layer: Y = MultiHead(RMSNorm(X)) + X, X' = SwiGLU(RMSNorm(Y)) + Y.

    x: [B, N, d_model] bf16 or fp32; module weights as in module_fwd (w_qkv, if given, is
    torch.cat([w_q, w_k, w_v], 1): one projection GEMM instead of three); w_gu: [d_model, 2*d_ff]
    gate and up weights interleaved by interleave_gate_up; w_down: [d_ff, d_model]; every weight
    bf16, or every weight fp16, and the GEMM operands take that type; norm weights fp32 [d_model],
    head_weight fp32 [Dv] (the per-head RMSNorm's gain). d_model a multiple of 256, d_ff of 128.
    Returns X' [B, N, d_model] fp32 (the residual stream is kept in fp32).

    Six launches: RMSNorm of X; the QKV projection; the fused attention; W_O with the residual
    add in its epilogue, which also writes Y (times norm2's gain) as the next operand and the row
    sums of Y^2; gate/up with SwiGLU in its epilogue, scaled by 1/RMS(Y) per row
    (RMSNorm(Y) W = (Y W) / r); W_down with the second residual add.

    Range: the 16-bit operand copy of Y (times norm2's gain) is taken before the
    normalisation, so fp16 weights need |Y * g| <= 65504; bf16 weights have fp32's range."""
    B, N, dm = x.shape
    M = B * N
    op = (w_qkv if w_qkv is not None else w_q).dtype
    _, n1 = add_rmsnorm(x, weight=norm1_weight, eps=eps, n_dtype=op, stream=stream)
    att = _module_attention(n1, w_q, w_k, w_v, n_heads, lam, lam_init, eps, head_weight, ws, stream, op, w_qkv)
    y, y16, sq = gemm_residual(att, w_o, x.reshape(M, dm), c16_dtype=op, c16_gain=norm2_weight, want_row_sq=True,
                               ws=ws, stream=stream)
    h = gemm_swiglu(y16, w_gu, row_sq=sq, sq_count=dm, eps=eps, out_dtype=op, ws=ws, stream=stream)
    out, _, _ = gemm_residual(h, w_down, y, ws=ws, stream=stream)
    return out.view(B, N, dm)


def gemm_residual(a, w, r, c16_dtype=None, c16_gain=None, want_row_sq=False, out=None, ws=None, stream=None):
    """C = a @ w + r in fp32: a [M, K] and w [K, N] both bf16 or both fp16 (contiguous rows),
    r [M, N] fp32, bf16 or fp16; N a multiple of 256. Optionally the 16-bit copy C * c16_gain
    (c16_dtype; c16_gain fp32 [N] or None) and row_sq [M, N // 256] (row sums of C^2 per
    256-column tile). Returns (C, C16 or None, row_sq or None)."""
    M, K = a.shape
    K2, N = w.shape
    if K2 != K or a.stride(1) != 1 or w.stride(1) != 1 or r.shape != (M, N) or r.stride(1) != 1:
        raise ValueError("a [M,K], w [K,N], r [M,N] with contiguous rows")
    if a.dtype != w.dtype or a.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("a and w must both be bf16 or both fp16")
    c = torch.empty((M, N), dtype=torch.float32, device=a.device) if out is None else out
    c16 = torch.empty((M, N), dtype=c16_dtype, device=a.device) if c16_dtype is not None else None
    sq = torch.empty((M, N // 256), dtype=torch.float32, device=a.device) if want_row_sq else None
    ws = workspace(256, a.device) if ws is None else ws
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    _check(load_library().diffattn_gemm_residual(
        ptr(a), ptr(w), ptr(r), ptr(c), ptr(c16), ptr(c16_gain), ptr(sq), M, N, K, a.stride(0), w.stride(0),
        r.stride(0), c.stride(0), c16.stride(0) if c16 is not None else 0, _dtype_code(a.dtype), _dtype_code(r.dtype),
        _dtype_code(c16_dtype) if c16_dtype is not None else 0, ptr(ws), ws.numel(), _stream_ptr(stream)),
        "diffattn_gemm_residual")
    return c, c16, sq


def gemm_swiglu(a, w_gu, row_sq=None, sq_count=None, eps: float = 1e-5, out_dtype=torch.float16, ws=None,
                stream=None):
    """H = SiLU(g / r) * (u / r): g, u the gate and up columns of a @ w_gu (w_gu [K, 2F] from
    interleave_gate_up), r = sqrt(sum(row_sq[m]) / sq_count + eps) per row (1 without row_sq).
    a and w_gu both bf16 or both fp16. Returns H [M, F] of out_dtype (bf16 or fp16)."""
    M, K = a.shape
    K2, F2 = w_gu.shape
    if K2 != K or a.stride(1) != 1 or w_gu.stride(1) != 1:
        raise ValueError("a [M,K] and w_gu [K,2F] with contiguous rows")
    h = torch.empty((M, F2 // 2), dtype=out_dtype, device=a.device)
    ws = workspace(256, a.device) if ws is None else ws
    n_sq = 0 if row_sq is None else row_sq.shape[1]
    if row_sq is not None and (row_sq.shape[0] != M or not row_sq.is_contiguous() or sq_count is None):
        raise ValueError("row_sq [M, n] contiguous, with sq_count")
    _check(load_library().diffattn_gemm_swiglu(
        ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(w_gu.data_ptr()), ctypes.c_void_p(h.data_ptr()),
        None if row_sq is None else ctypes.c_void_p(row_sq.data_ptr()), n_sq, float(sq_count or 1.0), float(eps), M,
        F2 // 2, K, a.stride(0), w_gu.stride(0), h.stride(0), _dtype_code(a.dtype), _dtype_code(out_dtype),
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_ptr(stream)), "diffattn_gemm_swiglu")
    return h


def gemm(a: torch.Tensor, w: torch.Tensor, out_dtype=torch.bfloat16, out=None, ws=None, stream=None):
    """C = a @ w with a [M,K] and w [K,N] row-major (unit last stride), both bf16 or both fp16;
    C fp32, bf16 or fp16."""
    M, K = a.shape
    K2, N = w.shape
    if K2 != K or a.stride(1) != 1 or w.stride(1) != 1:
        raise ValueError("a [M,K] and w [K,N] with contiguous rows")
    if a.dtype != w.dtype or a.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("a and w must both be bf16 or both fp16")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    ws = workspace(256, a.device) if ws is None else ws
    name = "diffattn_gemm_f16" if a.dtype == torch.float16 else "diffattn_gemm_bf16"
    _check(getattr(load_library(), name)(
        ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(out.data_ptr()), M, N, K,
        a.stride(0), w.stride(0), out.stride(0), _dtype_code(out.dtype), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        _stream_ptr(stream)), name)
    return out


gemm_bf16 = gemm


def module_fwd(x, w_q, w_k, w_v, w_o, n_heads: int, lam: float, lam_init: float, eps: float = 1e-5,
               norm_weight=None, ws=None, stream=None, out_dtype=torch.bfloat16, qkv_dtype=torch.float16,
               w_qkv=None):
    """Multi-head differential attention module: the projection GEMMs (one against
    w_qkv = torch.cat([w_q, w_k, w_v], 1) when it is given, else three), the fused
    attention reading Q/K/V in place through strided views, and the W_O GEMM.

    x [B,N,d_model]; w_q, w_k [d_model, h*2d]; w_v [d_model, h*Dv]; w_o [h*Dv, d_model],
    all bf16 or all fp16. Head i uses Q[..., 2di:2di+d] as Q1 and Q[..., 2di+d:2d(i+1)] as Q2
    (K likewise). The projections are written as qkv_dtype: fp16 by default (bf16
    rounding of Q, K and V alone would cost about 3e-3 relative error at the output);
    the attention output that W_O multiplies has the operands' type.

    Range: fp16 holds projections up to 65504 in magnitude; an entry beyond that
    overflows to infinity in the GEMM epilogue and the module's output is not
    finite. Inputs normalised before the projections (as in the layer) stay far
    inside it. Projections that large would also put the scores past the
    attention's own range (scaled scores below 2^28, see diffattn_fwd), so fp16 is
    no narrower in practice; qkv_dtype=torch.bfloat16 selects bf16 Q, K and V
    (8 significant bits instead of 11) for callers who want bf16 throughout.
    """
    att = _module_attention(x, w_q, w_k, w_v, n_heads, lam, lam_init, eps, norm_weight, ws, stream, x.dtype, w_qkv,
                            qkv_dtype)
    B, N, dm = x.shape
    y = gemm(att, w_o, out_dtype=out_dtype, ws=ws, stream=stream)
    return y.view(B, N, dm)


def _module_attention(x, w_q, w_k, w_v, n_heads, lam, lam_init, eps, norm_weight, ws, stream, att_dtype, w_qkv=None,
                      qkv_dtype=torch.float16):
    """The projections and the fused attention of module_fwd: returns concat(heads) [B*N, h*Dv]
    of att_dtype, the operand W_O multiplies."""
    if qkv_dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("qkv_dtype must be torch.float16 or torch.bfloat16")
    B, N, dm = x.shape
    h = n_heads
    x2 = x.reshape(B * N, dm)
    if w_qkv is not None:
        # one GEMM against [W_Q | W_K | W_V]; Q, K, V are column blocks of its output
        if w_q is not None:
            d, Dv = w_q.shape[1] // (2 * h), w_v.shape[1] // h
        else:
            raise ValueError("w_qkv also needs w_q and w_v (or their shapes) to split the heads")
        qkv = gemm(x2, w_qkv, out_dtype=qkv_dtype, ws=ws, stream=stream)
        c = qkv.shape[1]
        q, k, v = qkv[:, : 2 * d * h], qkv[:, 2 * d * h: 4 * d * h], qkv[:, 4 * d * h:]
        if c != 4 * d * h + Dv * h:
            raise ValueError("w_qkv must be torch.cat([w_q, w_k, w_v], 1)")
    else:
        d = w_q.shape[1] // (2 * h)
        Dv = w_v.shape[1] // h
        q = gemm(x2, w_q, out_dtype=qkv_dtype, ws=ws, stream=stream)
        k = gemm(x2, w_k, out_dtype=qkv_dtype, ws=ws, stream=stream)
        v = gemm(x2, w_v, out_dtype=qkv_dtype, ws=ws, stream=stream)
    # [B*N, h*2d] (column blocks, any row stride) -> [B, h, N, 2d] views, no copies
    q4 = q.unflatten(0, (B, N)).unflatten(2, (h, 2 * d)).permute(0, 2, 1, 3)
    k4 = k.unflatten(0, (B, N)).unflatten(2, (h, 2 * d)).permute(0, 2, 1, 3)
    v4 = v.unflatten(0, (B, N)).unflatten(2, (h, Dv)).permute(0, 2, 1, 3)
    att = diffattn_fwd(q4[..., :d], q4[..., d:], k4[..., :d], k4[..., d:], v4, lam, lam_init, eps, norm_weight,
                       out_dtype=att_dtype, ws=ws, stream=stream)
    return att.view(B * N, h * Dv)


_host_buffers = {}


def diffattn_fwd_host(q1, q2, k1, k2, v, lam, lam_init, eps=1e-5, out_dtype=torch.float32, device="cuda",
                      stream=None, out_host=None, chunks=None, norm_weight=None, causal=True):
    """End-to-end call from pinned HOST tensors [B,H,N,*] (contiguous); returns the host output
    [B,N,H,Dv]. One C-ABI call (diffattn_fwd_host): the work in `chunks` pieces (head ranges of
    one batch entry; default 4), each piece's copies in, prefill and copy back on three library
    streams, so the copies of one piece overlap the prefill and copies of others. The device staging buffer is allocated
    once per device and size, and reused; its first 256 bytes are the workspace, whose error word
    read_error(host_buffer_workspace(...)) reads. `stream` (default: the current one) waits for the
    last copy back, so synchronising it makes `out_host` valid."""
    names = (q1, q2, k1, k2, v)
    if any(t.is_cuda or not t.is_contiguous() or t.dtype != q1.dtype for t in names):
        raise ValueError("q1, q2, k1, k2, v: contiguous host tensors of one dtype")
    B, H, N, d = q1.shape
    Dv = v.shape[-1]
    dev = torch.device(device)
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if out_host is None:
        out_host = torch.empty((B, N, H, Dv), dtype=out_dtype, pin_memory=True)
    if out_host.shape != (B, N, H, Dv) or out_host.dtype != out_dtype or not out_host.is_contiguous():
        raise ValueError("out_host: contiguous [B, N, H, Dv] of out_dtype")
    buf = host_buffer_workspace(B, H, N, d, Dv, q1.dtype, out_dtype, dev)
    st = torch.cuda.current_stream(dev) if stream is None else stream
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    _check(load_library().diffattn_fwd_host(
        *(ptr(t) for t in names), ptr(out_host), ptr(norm_weight), B, H, N, d, Dv, int(bool(causal)), float(lam),
        float(lam_init), float(eps), _dtype_code(q1.dtype), _dtype_code(out_dtype), int(chunks or 0), ptr(buf),
        buf.numel(), _stream_ptr(st)), "diffattn_fwd_host")
    return out_host


def host_buffer_workspace(B, H, N, d, Dv, in_dtype, out_dtype, device):
    """The device staging buffer of diffattn_fwd_host for these sizes (cached per device: one
    buffer, regrown when a call needs more). Its first 256 bytes are the call's workspace."""
    n = ctypes.c_size_t()
    _check(load_library().diffattn_fwd_host_buffer_size(B, H, N, d, Dv, _dtype_code(in_dtype), _dtype_code(out_dtype),
                                                        ctypes.byref(n)), "diffattn_fwd_host_buffer_size")
    key = torch.device(device).index
    buf = _host_buffers.get(key)
    if buf is None or buf.numel() < n.value:
        buf = torch.zeros(n.value, dtype=torch.uint8, device=device)
        _host_buffers[key] = buf
    return buf

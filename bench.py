"""Benchmark of the differential-attention hot path on one GB300 (per rank).

A step is one pass of the prefill path over the B=4, H=16, N=2048, d=64,
Dv=128 bf16 workload (layer 6): lambda on the host, then the fused tcgen05
prefill kernel (both maps, combination, per-head RMSNorm, (1 - lambda_init)),
bf16 output. The headline value is algorithmic TFLOP/s: per (b, h),
4*Np*d + 2*Np*Dv with Np = N(N+1)/2 causal pairs. The decode path (64
sequences x 16 heads x 8192 cached tokens) is timed in the same run and
reported in the "decode" object as HBM GB/s over the KV-cache bytes.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Under torchrun each rank runs an independent replica (the path needs no
collective); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "DiffAttn fwd TFLOP/s & % GB300 BF16 peak; decode HBM GB/s & % peak"
PREFILL = "prefill_bf16"
DECODE = "decode_bf16"
NAMES = ("q1", "q2", "k1", "k2", "v")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def prefill_def_flops(w) -> float:
    n_pairs = w.N * (w.N + 1) / 2
    return w.B * w.H * (4 * n_pairs * w.d + 2 * n_pairs * w.Dv)


def prefill_exec_flops(w) -> float:
    n_pairs = w.N * (w.N + 1) / 2
    return w.B * w.H * (4 * n_pairs * w.d + 4 * n_pairs * w.Dv)


def prefill_bytes(w) -> int:
    """Inputs read once plus the bf16 output written once."""
    return w.B * w.H * w.N * (4 * w.d + w.Dv) * 2 + w.B * w.N * w.H * w.Dv * 2


def decode_kv_bytes(w) -> int:
    return w.B * w.H * w.N * (2 * w.d + w.Dv) * 2


CSRC = os.path.join(ROOT, "differential_attention_02_gb300", "csrc")


def profiled_traffic(key, files):
    """DRAM bytes per launch recorded from an ncu capture in profiles/traffic.json,
    or None when the kernel sources (its .cu file and common.cuh) have changed since
    that capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[key]
        h = hashlib.sha256()
        for name in files:
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(f.read())
    except (OSError, KeyError, ValueError):
        return None
    return rec["traffic_bytes"] if h.hexdigest()[:16] == rec["source_sha"] else None


def max_over_ranks(x: float, device="cpu") -> float:
    """The maximum of x over the ranks of the default process group (x itself
    without one): the job's step time is its slowest replica's."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job rate: the units all ranks processed divided by the slowest rank's time (per second)."""
    return world * units_per_rank / (ms_max * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples the SM clock and clock-event (throttle) reasons while the timed region runs.

    Reads NVML through ctypes every ~1 ms on a background thread (reading only;
    no GPU setting is changed). Falls back to `nvidia-smi -lms 200` when NVML
    cannot be loaded.
    """

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int):
        import threading
        self.gpu = gpu_index
        self.samples = []
        self.stop = threading.Event()
        self.thread = None
        self.max_mhz = None
        self.nvml = None
        self.proc = None

    def _open_nvml(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        getr = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = mx.value
        return nv, h, getr

    def _sample(self):
        import ctypes
        nv, h, getr = self.nvml
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        try:
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and getr(h, ctypes.byref(rs)) == 0:
                self.samples.append((mhz.value, rs.value))
        except (OSError, ctypes.ArgumentError):  # a failed read is a missing sample, not a failed run
            pass

    def _loop(self):
        while not self.stop.is_set():
            self._sample()
            time.sleep(0.001)

    def __enter__(self):
        import threading
        try:
            self.nvml = self._open_nvml()
            self._sample()  # one sample at the start of the region, whatever the thread manages
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
        except (OSError, AttributeError):
            self.nvml = None
            try:
                self.path = os.path.join("/tmp", f"diffattn_clocks_{os.getpid()}.csv")
                self.f = open(self.path, "w")
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                     "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                     "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
            except OSError:
                self.proc = None
        return self

    def __exit__(self, *a):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=2)
            self._sample()  # and one at its end, right after the closing synchronize
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait(timeout=5)
            self.f.close()

    def summary(self):
        if self.nvml is not None and self.samples:
            reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
            return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(self.samples), "source": "nvml"}
        if self.proc is not None:
            rows = []
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                try:
                    rows.append((float(parts[0]), float(parts[1]), parts[2:6]))
                except (ValueError, IndexError):
                    pass
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            if rows:
                return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                        "reasons": sorted({names[i] for _, _, f in rows for i, x in enumerate(f) if x == "Active"}),
                        "samples": len(rows), "source": "nvidia-smi"}
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"], "samples": 0}


# ----------------------------------------------------------------------------- reference arm (oracle)
def cpu_oracle_sample(budget_s: float):
    """Times the float64 oracle on whole heads of the prefill workload until budget_s is used."""
    from differential_attention_02_gb300 import inputs as gi
    from oracle import diffattn_oracle as orc

    w = gi.WORKLOADS[PREFILL]
    t = gi.prefill_inputs(w, B=1)  # batch row 0 of the workload
    lv = gi.lambda_vectors(w)
    lam, lam_init = orc.reparam_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer)
    per_head = prefill_def_flops(w) / (w.B * w.H)
    heads, t0 = 0, time.perf_counter()
    while True:
        h = heads % w.H
        o = orc.diffattn_head(*(t[k][0, h] for k in NAMES), lam)
        orc.head_rmsnorm_scale(o, lam_init, w.eps)
        heads += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return heads, el, heads * per_head / el / 1e12


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def run_reference(args, rank: int):
    if rank != 0:
        return
    for _ in range(args.warmup):
        cpu_oracle_sample(0.0)
    vals, total_heads, total_t = [], 0, 0.0
    for _ in range(args.steps):
        heads, el, tf = cpu_oracle_sample(args.ref_step_s)
        vals.append(tf)
        total_heads += heads
        total_t += el
    value = total_heads * prefill_def_flops_unit() / total_t / 1e12
    cores = cpu_threads()
    sample = (f"float64 NumPy oracle on whole heads (N=2048, d=64, Dv=128, causal) of the prefill workload, "
              f"{total_heads} heads in {args.steps} steps of >= {args.ref_step_s:.0f} s")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill B4 H16 N2048 d64 Dv128 causal, layer 6 (sampled heads)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def prefill_def_flops_unit():
    from differential_attention_02_gb300 import inputs as gi
    w = gi.WORKLOADS[PREFILL]
    return prefill_def_flops(w) / (w.B * w.H)


# ----------------------------------------------------------------------------- our arm
def run_e2e(args, da, w, host, lv, out_shape, dev, stream, world):
    """Same metric through the public API from pinned host buffers: H2D, prefill, D2H per step."""
    pin = {k: host[k].pin_memory() for k in NAMES}
    out_host = torch.empty(out_shape, dtype=torch.bfloat16, pin_memory=True)
    for _ in range(2):
        da.diffattn_fwd_host(*(pin[k] for k in NAMES), 0.5, 0.3, w.eps, out_dtype=torch.bfloat16,
                             device=dev, out_host=out_host)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        lam, lam_init = da.diffattn_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer)
        da.diffattn_fwd_host(*(pin[k] for k in NAMES), lam, lam_init, w.eps, out_dtype=torch.bfloat16,
                             device=dev, out_host=out_host)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    h2d = sum(pin[k].numel() * pin[k].element_size() for k in NAMES)
    d2h = out_host.numel() * out_host.element_size()
    # The copies alone, on one stream, with the same pinned buffers: what the host link allows.
    dbuf = {k: torch.empty_like(pin[k], device=dev) for k in NAMES}
    dout = torch.empty(out_shape, dtype=torch.bfloat16, device=dev)

    def copies(h2d_on, d2h_on):
        for _ in range(max(3, args.steps)):
            if h2d_on:
                for k in NAMES:
                    dbuf[k].copy_(pin[k], non_blocking=True)
            if d2h_on:
                out_host.copy_(dout, non_blocking=True)

    timing = {}
    for name, a, b in (("h2d", True, False), ("d2h", False, True), ("both", True, True)):
        copies(a, b)  # warm-up
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        copies(a, b)
        c1.record(stream)
        torch.cuda.synchronize()
        timing[name] = c0.elapsed_time(c1) / max(3, args.steps)
    return {"value": world * prefill_def_flops(w) / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies_alone": {
                "note": "the step's host<->device copies alone, one stream, same pinned buffers",
                "h2d_ms": timing["h2d"], "h2d_gbs": h2d / (timing["h2d"] * 1e-3) / 1e9,
                "d2h_ms": timing["d2h"], "d2h_gbs": d2h / (timing["d2h"] * 1e-3) / 1e9,
                "h2d_then_d2h_ms": timing["both"],
                "e2e_over_copies": e2e_ms / timing["both"]}}


def time_device(fn, steps, warmup, stream, flush=None):
    """Median CUDA-event time (ms) of fn() over `steps` calls after `warmup` calls,
    each call bracketed by its own pair of events on `stream`; with `flush`, L2 is
    evicted (untimed) before each timed call."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        if flush is not None:
            flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def extra_reps(args) -> int:
    """Timed calls per extra workload: at least 20, more when the run asks for more steps."""
    return max(20, args.steps)


def run_long_prefill(args, da, gi, dev, stream, peaks, peak_kind):
    """The B=1, H=16, N=16384 prefill workload (layer 12), bf16 in/out."""
    w = gi.WORKLOADS["long_prefill_bf16"]
    x = {k: v.to(dev) for k, v in gi.prefill_inputs(w).items()}
    lv = gi.lambda_vectors(w)
    lam, lam_init = da.diffattn_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer)
    out = torch.empty((w.B, w.N, w.H, w.Dv), dtype=torch.bfloat16, device=dev)
    ws = da.workspace(256, dev)
    fn = lambda: da.diffattn_fwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, lam_init, w.eps,
                                 out_dtype=torch.bfloat16, out=out, ws=ws, stream=stream)
    ms = time_device(fn, extra_reps(args), args.warmup, stream)
    assert da.read_error(ws) == 0
    tf = prefill_def_flops(w) / (ms * 1e-3) / 1e12
    return {"workload": "prefill B1 H16 N16384 d64 Dv128 causal, layer 12, bf16 in/out", "ms_per_step": ms,
            "value": tf, "unit": "TFLOP/s", "exec_tflops": prefill_exec_flops(w) / (ms * 1e-3) / 1e12,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "peak_kind": f"{peak_kind} bf16 burst"},
            "gpu_launches_per_step": 1}


def run_module(args, da, gi, dev, stream, peaks, peak_kind):
    """Multi-head DiffAttn module: X [2,4096,2048] -> the Q/K/V projections (one GEMM against
    [W_Q | W_K | W_V], concatenated once, untimed), attention (h=8, d=128, Dv=256), W_O;
    layer 1 (the layer changes only lambda/lambda_init)."""
    w = gi.WORKLOADS["module_bf16"]
    t = {k: v.to(dev) for k, v in gi.module_inputs(w).items()}
    wqkv = torch.cat([t["w_q"], t["w_k"], t["w_v"]], dim=1).contiguous()
    lv = gi.lambda_vectors(w)
    lam, lam_init = da.diffattn_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], 1)
    ws = da.workspace(256, dev)
    fn = lambda: da.module_fwd(t["x"], t["w_q"], t["w_k"], t["w_v"], t["w_o"], w.H, lam, lam_init, w.eps, ws=ws,
                               stream=stream, w_qkv=wqkv)
    ms = time_device(fn, extra_reps(args), args.warmup, stream)
    assert da.read_error(ws) == 0
    n_pairs = w.N * (w.N + 1) / 2
    att = w.B * w.H * (4 * n_pairs * w.d + 2 * n_pairs * w.Dv)
    M = w.B * w.N
    gemm = 2.0 * M * w.d_model * (2 * w.H * 2 * w.d + w.H * w.Dv) + 2.0 * M * w.H * w.Dv * w.d_model
    tf = (att + gemm) / (ms * 1e-3) / 1e12
    return {"workload": "module X[2,4096,2048], h8 d128 Dv256, causal, layer 1; bf16 weights, fp16 Q/K/V",
            "ms_per_step": ms, "value": tf, "unit": "TFLOP/s", "flops_per_step": att + gemm,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "peak_kind": f"{peak_kind} bf16 burst"},
            "gpu_launches_per_step": 3}


def run_layer(args, da, gi, dev, stream, peaks, peak_kind):
    """One DIFF Transformer layer on X [2,4096,2048]: pre-RMSNorm, the module above,
    residual add + RMSNorm, the SwiGLU FFN (d_ff 5632) and the second residual add, in six
    launches (the residual adds, the second RMSNorm and SwiGLU run in GEMM epilogues)."""
    w = gi.WORKLOADS["layer_bf16"]
    # Weights as fp16 copies of the bf16 draws (exact above 2^-14 in magnitude; the ~0.3% of
    # smaller values move by at most 2^-25), so the GEMM operands are fp16 as well.
    t = {k: (v.to(dev).half() if k.startswith("w_") else v.to(dev)) for k, v in gi.layer_inputs(w).items()}
    # one-time weight layouts (untimed): gate/up interleaved for the SwiGLU epilogue, [W_Q | W_K | W_V]
    wgu = da.interleave_gate_up(t.pop("w_gate"), t.pop("w_up"))
    wqkv = torch.cat([t["w_q"], t["w_k"], t["w_v"]], dim=1).contiguous()
    lv = gi.lambda_vectors(w)
    lam, lam_init = da.diffattn_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer)
    ws = da.workspace(256, dev)
    fn = lambda: da.layer_fwd(t["x"], t["w_q"], t["w_k"], t["w_v"], t["w_o"], wgu, t["w_down"], w.H, lam, lam_init,
                              w.eps, ws=ws, stream=stream, w_qkv=wqkv)
    ms = time_device(fn, extra_reps(args), args.warmup, stream)
    assert da.read_error(ws) == 0
    n_pairs = w.N * (w.N + 1) / 2
    att = w.B * w.H * (4 * n_pairs * w.d + 2 * n_pairs * w.Dv)
    M = w.B * w.N
    gemm = 2.0 * M * w.d_model * (2 * w.H * 2 * w.d + w.H * w.Dv) + 2.0 * M * w.H * w.Dv * w.d_model
    ffn = 6.0 * M * w.d_model * w.d_ff
    tf = (att + gemm + ffn) / (ms * 1e-3) / 1e12
    return {"workload": "layer X[2,4096,2048], h8 d128 Dv256, SwiGLU d_ff 5632, causal, layer 1; fp16 copies of "
                        "bf16 weights, fp16 GEMM operands, fp32 residual stream",
            "ms_per_step": ms, "value": tf, "unit": "TFLOP/s", "flops_per_step": att + gemm + ffn,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "peak_kind": f"{peak_kind} bf16 burst"},
            "gpu_launches_per_step": 6}


def run_backward(args, da, gi, dev, stream, peaks, peak_kind):
    """The backward pass on the prefill workload, bf16 inputs, fp32 gradients: from the state the
    training forward saved (diffattn_fwd_train + diffattn_bwd(saved=...)), and, beside it, the
    backward that re-runs the forward itself (diffattn_bwd alone) and the two forwards' times."""
    w = gi.WORKLOADS["prefill_bf16"]
    x = {k: v.to(dev) for k, v in gi.prefill_inputs(w).items()}
    dy = gi.output_grad(w).to(dev)
    lv = gi.lambda_vectors(w)
    lam, lam_init = da.diffattn_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer)
    ops = (x["q1"], x["q2"], x["k1"], x["k2"], x["v"])
    ws = da.workspace(da.bwd_workspace_bytes(w.B, w.H, w.N, w.d, w.Dv), dev)
    out = torch.empty((w.B, w.N, w.H, w.Dv), dtype=torch.bfloat16, device=dev)
    fws = da.workspace(256, dev)
    saved = da.saved_state(w.B, w.H, w.N, w.Dv, dev)
    train = lambda: da.diffattn_fwd_train(*ops, lam, lam_init, w.eps, out_dtype=torch.bfloat16, out=out,
                                          saved=saved, ws=fws, stream=stream)
    plain = lambda: da.diffattn_fwd(*ops, lam, lam_init, w.eps, out_dtype=torch.bfloat16, out=out, ws=fws,
                                    stream=stream)
    ms_train = time_device(train, extra_reps(args), args.warmup, stream)
    ms_plain = time_device(plain, extra_reps(args), args.warmup, stream)
    train()  # the saved state of these inputs
    from_saved = lambda: da.diffattn_bwd(*ops, dy, lam, lam_init, w.eps, want_dnorm_weight=True, ws=ws,
                                         stream=stream, saved=saved)
    recompute = lambda: da.diffattn_bwd(*ops, dy, lam, lam_init, w.eps, want_dnorm_weight=True, ws=ws,
                                        stream=stream)
    ms = time_device(from_saved, extra_reps(args), args.warmup, stream)
    ms_re = time_device(recompute, extra_reps(args), args.warmup, stream)
    assert da.read_error(ws) == 0 and da.read_error(fws) == 0
    n_pairs = w.N * (w.N + 1) / 2
    # Chain-rule FLOPs per (b, h): per map S recomputed, dQ and dK (2 Np d each); dV and dA (2 Np Dv each).
    flops = w.B * w.H * (12 * n_pairs * w.d + 4 * n_pairs * w.Dv)
    # Executed on the tensor cores: the key-side kernel (S1, S2, dA, dV, dK1, dK2: 8 Np d + 4 Np Dv) and the
    # query-side one (S1, S2, dA, dQ1, dQ2: 8 Np d + 2 Np Dv); re-running the forward adds 4 Np d + 4 Np Dv.
    exec_flops = w.B * w.H * n_pairs * (16 * w.d + 6 * w.Dv)
    exec_re = w.B * w.H * n_pairs * (20 * w.d + 10 * w.Dv)
    tf = flops / (ms * 1e-3) / 1e12
    tf_re = flops / (ms_re * 1e-3) / 1e12
    return {"workload": "backward of the prefill workload B4 H16 N2048 d64 Dv128 causal, bf16 in, fp32 gradients, "
                        "from the training forward's saved state (x = O1/l1 - lambda O2/l2 in fp32, O2/l2 in the operand "
                        "type, each map's row log-sum-exp)",
            "ms_per_step": ms, "value": tf, "unit": "TFLOP/s", "flops_per_step": flops,
            "exec_tflops": exec_flops / (ms * 1e-3) / 1e12,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "peak_kind": f"{peak_kind} bf16 burst",
                         "traffic_dominant_kernel": {
                             "kernel": "bwd_dkdv_kernel",
                             "bytes": profiled_traffic("bwd_dkdv_prefill_B4H16N2048", ["bwd_tcgen05.cu", "common.cuh"])}},
            "gpu_launches_per_step": 4,
            "recompute": {"note": "diffattn_bwd without saved state: the forward re-run as its first launch",
                          "ms_per_step": ms_re, "value": tf_re, "frac": tf_re / peaks["bf16_tflops"],
                          "exec_tflops": exec_re / (ms_re * 1e-3) / 1e12, "gpu_launches_per_step": 4},
            "forward": {"note": "the same inputs' forward, bf16 out: diffattn_fwd_train (per-tile kernel, saves "
                                f"{da.train_saved_bytes(w.B, w.H, w.N, w.Dv) / 1e6:.0f} MB of state) against diffattn_fwd",
                        "train_ms": ms_train, "plain_ms": ms_plain}}


def run_decode(args, da, gi, dev, stream, peaks, peak_kind):
    """Times the split-KV decode (split kernel + merge kernel) on the decode workload."""
    import dataclasses
    wd = gi.WORKLOADS[DECODE]
    if args.decode_batch:
        wd = dataclasses.replace(wd, B=args.decode_batch)
    hd = gi.decode_inputs(wd)
    lvd = gi.lambda_vectors(wd)
    y = {k: hd[k].to(dev) for k in NAMES}
    del hd
    dout = torch.empty((wd.B, wd.H, wd.Dv), dtype=torch.bfloat16, device=dev)
    dws = da.workspace(da.decode_workspace_bytes(wd.B, wd.H, wd.N, wd.d, wd.Dv), dev)
    lam, lam_init = da.diffattn_lambda(lvd["lq1"], lvd["lk1"], lvd["lq2"], lvd["lk2"], wd.layer)

    def dstep():
        da.diffattn_decode(y["q1"], y["q2"], y["k1"], y["k2"], y["v"], lam, lam_init, eps=wd.eps,
                           out_dtype=torch.bfloat16, out=dout, ws=dws, stream=stream)

    for _ in range(max(3, args.warmup)):
        dstep()
    torch.cuda.synchronize()
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    for i in range(args.steps):
        dev_ev[i][0].record(stream)
        dstep()
        dev_ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert da.read_error(dws) == 0
    dms = statistics.median(a.elapsed_time(b) for a, b in dev_ev)
    kvb = decode_kv_bytes(wd)
    gbs = kvb / (dms * 1e-3) / 1e9
    per_seq = profiled_traffic("decode_split_per_sequence_H16L8192", ["decode_bf16.cu", "common.cuh"])
    traffic = per_seq * wd.B if (per_seq is not None and wd.H == 16 and wd.N == 8192) else None
    serving = run_serving(args, da, wd, y, lam, lam_init, dev, stream, peaks, kvb)
    return {"workload": f"decode {wd.B} seqs x 1 token, H{wd.H}, L{wd.N}, d{wd.d}, Dv{wd.Dv}, layer {wd.layer}",
            "ms_per_step": dms, "value": gbs, "unit": "GB/s", "kv_bytes_per_step": kvb,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": traffic, "peak_kind": peak_kind,
                         "frac_of_spec_8tbs": gbs / 8000.0},
            "gpu_launches_per_step": 2, "serving": serving}


def run_serving(args, da, wd, y, lam, lam_init, dev, stream, peaks, kvb):
    """The decode workload as a serving step over a paged KV cache: the same caches
    scattered into shuffled 64-token pages; each step appends every sequence's new
    token (position L-1) and decodes."""
    B, H, L = wd.B, wd.H, wd.N
    maxp = L // 64
    g = torch.Generator(device="cpu").manual_seed(17)
    table = torch.randperm(B * maxp, generator=g).view(B, maxp).to(torch.int32).to(dev)
    pools = {}
    for k in ("k1", "k2", "v"):
        c = y[k]
        pool = torch.empty(B * maxp, H, 64, c.shape[-1], dtype=c.dtype, device=dev)
        pool[table.view(-1).long()] = c.view(B, H, maxp, 64, -1).permute(0, 2, 1, 3, 4).reshape(B * maxp, H, 64, -1)
        pools[k] = pool
    new = {k: y[k][:, :, L - 1].contiguous() for k in ("k1", "k2", "v")}
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    out = torch.empty((B, H, wd.Dv), dtype=torch.bfloat16, device=dev)
    ws = da.workspace(da.decode_workspace_bytes(B, H, L, wd.d, wd.Dv), dev)

    def step():
        da.diffattn_kv_append_paged(new["k1"], new["k2"], new["v"], pools["k1"], pools["k2"], pools["v"], table,
                                    lens, stream=stream)
        da.diffattn_decode_paged(y["q1"], y["q2"], pools["k1"], pools["k2"], pools["v"], table, lens, lam,
                                 lam_init, L=L, eps=wd.eps, out_dtype=torch.bfloat16, out=out, ws=ws, stream=stream)

    ms = time_device(step, extra_reps(args), max(3, args.warmup), stream)
    assert da.read_error(ws) == 0
    gbs = kvb / (ms * 1e-3) / 1e9
    res = {"workload": f"decode {B} seqs, H{H}, L{L}: new token appended to a paged KV cache (64-token pages, "
                       f"shuffled) then decoded", "ms_per_step": ms, "value": gbs, "unit": "GB/s",
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"], "frac_of_spec_8tbs": gbs / 8000.0},
           "gpu_launches_per_step": 3}

    # The same serving step over an fp8 (e4m3) cache: one scale per tensor (amax / 448), the
    # pages quantized once here (setup, untimed); the append quantizes the new token.
    scales = tuple(float(pools[k].abs().max().float()) / 448.0 for k in ("k1", "k2", "v"))
    q8 = {}
    for k, sc in zip(("k1", "k2", "v"), scales):
        q8[k] = (pools[k].float() / sc).to(torch.float8_e4m3fn)
        pools[k] = None
    del pools

    def step8():
        da.diffattn_kv_append_paged(new["k1"], new["k2"], new["v"], q8["k1"], q8["k2"], q8["v"], table, lens,
                                    stream=stream, scales=scales)
        da.diffattn_decode_paged(y["q1"], y["q2"], q8["k1"], q8["k2"], q8["v"], table, lens, lam, lam_init, L=L,
                                 eps=wd.eps, out_dtype=torch.bfloat16, out=out, ws=ws, stream=stream, scales=scales)

    ms8 = time_device(step8, extra_reps(args), max(3, args.warmup), stream)
    assert da.read_error(ws) == 0
    gbs8 = kvb / 2 / (ms8 * 1e-3) / 1e9
    per_seq8 = profiled_traffic("decode_split_fp8_per_sequence_H16L8192", ["decode_bf16.cu", "common.cuh"])
    res["fp8_cache"] = {
        "workload": "the same serving step with the K1, K2, V pages in fp8 e4m3 (one scale per tensor)",
        "ms_per_step": ms8, "value": gbs8, "unit": "GB/s", "kv_bytes_per_step": kvb // 2,
        "speedup_vs_bf16_cache": ms / ms8,
        "roofline": {"bound": "hbm", "achieved": gbs8, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs8 / peaks["hbm_gbs"],
                     "traffic": per_seq8 * B if (per_seq8 is not None and H == 16 and L == 8192) else None},
        "gpu_launches_per_step": 3}
    del q8
    return res


def run_ours(args, rank: int, world: int, local_rank: int):
    import differential_attention_02_gb300 as da
    from differential_attention_02_gb300 import build as dab
    from differential_attention_02_gb300 import inputs as gi

    dab.build()
    da.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    peaks, peak_kind = load_peaks()

    if args.only:  # one section alone (profiling): no headline line
        fn = {"decode": run_decode, "long_prefill": run_long_prefill, "module": run_module, "layer": run_layer,
              "backward": run_backward}[args.only]
        res = fn(args, da, gi, dev, stream, peaks, peak_kind)
        if rank == 0:
            print(json.dumps({"only": args.only, "result": res}), flush=True)
        return

    # -------- inputs resident in HBM
    w = gi.WORKLOADS[PREFILL]
    host = gi.prefill_inputs(w)
    lv = gi.lambda_vectors(w)
    x = {k: host[k].to(dev) for k in NAMES}
    out = torch.empty((w.B, w.N, w.H, w.Dv), dtype=torch.bfloat16, device=dev)
    ws = da.workspace(256, dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > 129 MB L2

    def step():
        lam, lam_init = da.diffattn_lambda(lv["lq1"], lv["lk1"], lv["lq2"], lv["lk2"], w.layer)
        da.diffattn_fwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, lam_init, w.eps,
                        out_dtype=torch.bfloat16, out=out, ws=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert da.read_error(ws) == 0

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        barrier()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()  # evict L2 between timed steps (not timed)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        barrier()
        t_wall = time.perf_counter() - t_wall
    clocks = clk.summary()
    ms = [a.elapsed_time(b) for a, b in ev]
    ms_step = max_over_ranks(sum(ms) / len(ms), dev)
    ms_median = max_over_ranks(statistics.median(ms), dev)
    flops = prefill_def_flops(w)
    value = job_throughput(flops, ms_step, world) / 1e12
    achieved = flops / (ms_step * 1e-3) / 1e12  # the prefill kernel is the whole step on the GPU
    assert da.read_error(ws) == 0

    # -------- end to end from pinned host buffers through the public API
    e2e = None
    if not args.skip_e2e:
        e2e = run_e2e(args, da, w, host, lv, out.shape, dev, stream, world)
    del x, out

    # -------- decode workload (HBM bound; 4.3 GB of KV cache, larger than L2)
    dec = None
    if not args.skip_decode:
        dec = run_decode(args, da, gi, dev, stream, peaks, peak_kind)
    # -------- the other workloads, reported beside the headline
    extra = {}
    if not args.skip_extra:
        extra["long_prefill"] = run_long_prefill(args, da, gi, dev, stream, peaks, peak_kind)
        extra["module"] = run_module(args, da, gi, dev, stream, peaks, peak_kind)
        extra["layer"] = run_layer(args, da, gi, dev, stream, peaks, peak_kind)
        extra["backward"] = run_backward(args, da, gi, dev, stream, peaks, peak_kind)
    if rank != 0:
        return
    cpu = None
    if not args.skip_cpu_baseline and world == 1:
        heads, el, tf = cpu_oracle_sample(args.cpu_budget_s)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{heads} whole heads (N=2048, d=64, Dv=128, causal) of the prefill workload, "
                         f"float64 NumPy, {el:.1f} s"}
    peak = peaks["bf16_tflops"]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill B4 H16 N2048 d64 Dv128 causal, layer 6, bf16 in/out, fp32 accumulate",
                   "l2": "flushed between timed steps (256 MB write, untimed)",
                   "flops": "algorithmic: 4*Np*d + 2*Np*Dv per (b,h), Np = N(N+1)/2",
                   "exec_tflops": world * prefill_exec_flops(w) / (ms_step * 1e-3) / 1e12,
                   "ms_per_step_median": ms_median,
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} bf16 burst",
                     "kernel": "fwd_persist_kernel<64, 128> (one CTA per SM walking the query tiles)",
                     "traffic": profiled_traffic("fwd_persist_prefill_B4H16N2048", ["fwd_tcgen05.cu", "common.cuh"]),
                     "algorithmic_bytes": prefill_bytes(w)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "decode": dec,
        **extra,
        "clocks": clocks,
        "gpu_launches": args.steps,
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-extra", action="store_true", help="skip the long-prefill and module lines")
    ap.add_argument("--decode-batch", type=int, default=0, help="override the decode workload's batch (profiling)")
    ap.add_argument("--only", default="", choices=["", "decode", "long_prefill", "module", "layer", "backward"],
                    help="run one section alone and print its result (profiling), not the bench line")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-step-s", type=float, default=8.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

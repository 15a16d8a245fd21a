"""Host-side logic of bench.py, no GPU: the max-over-ranks reduction of the
replica path on two gloo ranks, and the reference arm's JSON line."""

import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 1.0 + rank  # rank 1 is the slow replica
    m = bench.max_over_ranks(ms, "cpu")
    out[rank] = (m, bench.job_throughput(10.0, m, world))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_on_two_gloo_ranks():
    manager = mp.get_context("spawn").Manager()  # no fork of this multi-threaded process
    out = manager.dict()
    port = 29500 + os.getpid() % 1000
    mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == (2.0, 2 * 10.0 / 2e-3)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(5.0, 10.0, 1) == 500.0


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                        "--ref-step-s", "0.2"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_sampler_brackets_the_region_with_a_fake_nvml(monkeypatch):
    """The NVML path on a stand-in library: samples at the start and end of the region
    (plus whatever the thread adds), median clock, and throttle reasons decoded."""
    import ctypes

    class FakeNvml:
        def __init__(self):
            self.calls = 0

        def nvmlDeviceGetClockInfo(self, h, kind, out):
            self.calls += 1
            ctypes.cast(out, ctypes.POINTER(ctypes.c_uint))[0] = 1900 + 10 * (self.calls % 3)
            return 0

    fake = FakeNvml()

    def reasons(h, out):
        ctypes.cast(out, ctypes.POINTER(ctypes.c_ulonglong))[0] = 0x4  # sw_power_cap
        return 0

    def fake_open(self):
        self.max_mhz = 2070
        return fake, None, reasons

    monkeypatch.setattr(bench.ClockSampler, "_open_nvml", fake_open)
    with bench.ClockSampler(0) as clk:
        pass
    out = clk.summary()
    assert out["source"] == "nvml" and out["samples"] >= 2
    assert out["sm_max_mhz"] == 2070 and 1900 <= out["sm_mhz"] <= 1920
    assert out["reasons"] == ["sw_power_cap"]

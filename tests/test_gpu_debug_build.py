"""The debug build (libdiffattn_debug.so, device-side index checks) on the GPU.

compute-sanitizer is not available on the GPU pool, so a build compiled with
DIFFATTN_DEBUG_CHECKS stands in for it: its kernels check the TMA coordinates
of the tensor-core prefill and GEMM, the paged block-table entries and the
split ranges of the decode, and record a failure in the error word (kind 2)
instead of trapping. Here the small and ragged parity tests run once against
that build (each of them asserts that the error word stays zero), and a
block-table entry outside the page pool is shown to be reported by the debug
build's check (which then reads page 0 in its place, so no access leaves the
pool).
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# The small and ragged shapes of the parity suite: prefill (one-CTA and CTA-pair
# kernels), decode (contiguous, paged, shared KV heads, append, fp8), GEMM.
SUBSET = [
    "tests/test_gpu_prefill.py::test_bf16_prefill_small_and_ragged",
    "tests/test_gpu_prefill.py::test_bf16_lambda_values",
    "tests/test_gpu_decode.py::test_decode_small",
    "tests/test_gpu_decode.py::test_decode_ragged_lengths_ignore_stale_cache",
    "tests/test_gpu_decode.py::test_decode_split_count_invariance",
    "tests/test_gpu_decode.py::test_paged_decode_matches_contiguous_and_oracle",
    "tests/test_gpu_decode.py::test_paged_decode_grouped_kv_heads",
    "tests/test_gpu_decode.py::test_kv_append_paged_then_decode",
    "tests/test_gpu_decode_fp8.py",
    "tests/test_gpu_gemm.py",
    "tests/test_gpu_module.py::test_module_reduced_length",
]

# A paged decode whose block table points one sequence at a page past the pool
# (run against the debug build only, whose check turns the entry into an error).
PROBE = r"""
import torch
import differential_attention_02_gb300 as da
da.load_library()
H, d, Dv, P = 2, 64, 128, 4
g = torch.Generator().manual_seed(5)
pages = {k: torch.randn(P, H, 64, Dv if k == "v" else d, generator=g).to(torch.bfloat16).cuda() for k in ("k1", "k2", "v")}
q = {k: torch.randn(1, H, d, generator=g).to(torch.bfloat16).cuda() for k in ("q1", "q2")}
table = torch.tensor([[0, P + 3]], dtype=torch.int32).cuda()   # second page outside the pool
lens = torch.tensor([100], dtype=torch.int32).cuda()
ws = da.workspace(da.decode_workspace_bytes(1, H, 128, d, Dv, 1))
da.diffattn_decode_paged(q["q1"], q["q2"], pages["k1"], pages["k2"], pages["v"], table, lens, 0.3, 0.2, L=128,
                         num_splits=1, ws=ws)
print("CODE", da.read_error(ws))
"""


@pytest.fixture(scope="module")
def libs():
    from differential_attention_02_gb300 import build
    return build.build(), build.build(debug=True)


def _env(lib):
    return dict(os.environ, DIFFATTN_LIBRARY=lib)


def test_small_and_ragged_parity_under_debug_build(libs):
    _, debug = libs
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider", *SUBSET],
                       cwd=ROOT, env=_env(debug), capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


def test_out_of_range_page_is_reported_by_the_debug_build(libs):
    _, debug = libs
    r = subprocess.run([sys.executable, "-c", PROBE], cwd=ROOT, env=_env(debug), capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    code = int(r.stdout.split("CODE")[-1])
    assert code == (0xA1 << 8) | 2  # site of the block-table check, kind 2 = index

"""The in-kernel split-KV merge's bookkeeping, checked on the host (no GPU).

`merge_bookkeeping_check.cu` includes the decode path's schedule header and
calls its real share arithmetic and `cut_piece` on thousands of random call
shapes (short, decode-like, mixed and very long segments; 1 to 2048
workers), asserting that every arrival counter belongs to one segment and
receives exactly its total, and that every fold reads the slots the pieces
were written to. nvcc builds it for the host here; the test is skipped
where nvcc is missing."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


def test_merge_counters_and_slots_on_random_call_shapes(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "merge_bookkeeping_check")
    build = subprocess.run(
        [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
         "--expt-relaxed-constexpr", "-O2",
         "-I", os.path.join(ROOT, "paged_kv_cache_154_gb300", "csrc"),
         os.path.join(ROOT, "tests", "merge_bookkeeping_check.cu"), "-o", exe],
        capture_output=True, text=True, timeout=600)
    assert build.returncode == 0, build.stderr[-2000:]
    run = subprocess.run([exe, "3000"], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0 and run.stdout.startswith("ok"), run.stdout[-2000:]

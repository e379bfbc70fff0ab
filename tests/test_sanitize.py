"""The host block pool (csrc/pool.cpp) and the CPU oracle (oracle/oracle.c)
under AddressSanitizer and UndefinedBehaviorSanitizer, no GPU.

`sanitize_check.cpp` compiles the pool source into a standalone program with
g++ -fsanitize=address,undefined, links the oracle built the same way with
gcc, and replays seeded random traces of every pool call -- forks, appends
by slots and by token ids with the prefix cache off and at three LRU sizes,
copy-on-write, frees (and double frees), fork groups, argument errors --
checking the pool's counts after each step, then runs the oracle's
attention, quantiser, appends and block copies on small caches of every
element type. Any out-of-bounds access, use after free, leak or undefined
operation stops the program with a report."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SAN = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer",
       "-g", "-O1"]


def _cuda_include():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "include", "cuda.h")):
            return os.path.join(c, "include")
    return None


def test_pool_and_oracle_under_asan_ubsan(tmp_path):
    if shutil.which("g++") is None or shutil.which("gcc") is None:
        pytest.skip("gcc/g++ not available")
    inc = _cuda_include()
    if inc is None:
        pytest.skip("CUDA headers not available (the pool's header includes them)")
    orc = str(tmp_path / "oracle.o")
    exe = str(tmp_path / "sanitize_check")
    r = subprocess.run(["gcc", "-c", "-std=c11", "-ffp-contract=off", "-fopenmp"] + SAN +
                       [os.path.join(ROOT, "oracle", "oracle.c"), "-o", orc],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run(["g++", "-std=c++17", "-fopenmp"] + SAN +
                       ["-I", os.path.join(ROOT, "paged_kv_cache_154_gb300", "csrc"), "-I", inc,
                        os.path.join(ROOT, "tests", "sanitize_check.cpp"), orc, "-lm", "-o", exe],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    env = dict(os.environ, ASAN_OPTIONS="abort_on_error=0:halt_on_error=1:detect_leaks=1",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    run = subprocess.run([exe, "1500"], capture_output=True, text=True, timeout=600, env=env)
    out = run.stdout + run.stderr
    if "LeakSanitizer does not work under ptrace" in out:   # some sandboxes forbid it
        env["ASAN_OPTIONS"] = "abort_on_error=0:halt_on_error=1:detect_leaks=0"
        run = subprocess.run([exe, "1500"], capture_output=True, text=True, timeout=600, env=env)
        out = run.stdout + run.stderr
    assert run.returncode == 0 and run.stdout.startswith("ok"), out[-3000:]
    # the traces reached the paths they are meant to exercise
    import re
    n = [int(x) for x in re.findall(r"(\d+) ", run.stdout)[:4]]
    assert n[0] >= 7000 and n[1] > 0 and n[2] > 0 and n[3] > 0, run.stdout

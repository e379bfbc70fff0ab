"""A bounded wait that runs out, on the GPU, without faulting it.

Every wait in the decode kernels is bounded: after a time limit it records
a code in the device error word, the kernel drains its copies in flight and
returns, and the context stays usable. This test builds a separate copy of
the library (libpa_waittest.so, the product libpa.so is not touched) with
a 1 ms limit and a test hook that makes the balanced kernel's first worker
skip issuing the copy of one of its blocks -- a copy that is simply never
started, so the wait for it cannot complete. The call must come back with
PA_DEVERR_WAIT_FULL in the error word; after the workspace's arrival
counters are zeroed again (the library's rule after an error), the next
call with the hook off must match the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
import paged_kv_cache_154_gb300 as pa
from gpu_harness import check_out, run_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def test_lib():
    from paged_kv_cache_154_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    path = build.build_variant("pa_waittest", ["-DPA_TEST_HOOKS", "-DPA_WAIT_LIMIT_NS=1000000ull"])
    L = ctypes.CDLL(path)
    for name, (args, res) in pa._SIGS.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    L.pa_test_skip_copy.argtypes = [ctypes.c_int]
    L.pa_test_skip_copy.restype = ctypes.c_int
    return L


def test_wait_that_runs_out_is_reported_and_the_next_call_is_correct(test_lib, monkeypatch):
    wl = W.simple("wait_limit", 808, [300, 1000, 700, 2500], [1, 1, 1, 1], 32, 8, 128, "bf16")
    ref, cache, si, out = run_both(wl)                # the product library, for reference
    monkeypatch.setattr(pa, "_lib", test_lib)         # every binding call now goes to the test copy
    args = (si.q, cache.k, cache.v, si.block_tables, si.context_lens, si.max_context_len, wl.scale,
            None, 1, cache.num_blocks)
    assert test_lib.pa_test_skip_copy(0) == 0         # worker 0 never issues its first block
    got = torch.zeros_like(si.out)
    pa.decode(got, *args, workspace=si.workspace)
    torch.cuda.synchronize()                          # the kernel came back
    code = pa.device_error()
    assert code & pa.DEVERR_WAIT_FULL, hex(code)
    assert not code & (pa.DEVERR_BAD_BLOCK | pa.DEVERR_BAD_SLOT), hex(code)
    # hook off, counters zeroed again: the same call is correct
    assert test_lib.pa_test_skip_copy(-1) == 0
    si.workspace[:pa.ARRIVAL_BYTES].zero_()
    got.fill_(float("nan"))
    pa.decode(got, *args, workspace=si.workspace)
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    check_out(ref, got, "bf16")

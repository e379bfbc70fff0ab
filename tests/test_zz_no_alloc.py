"""pa_decode_no_alloc against pa_decode and the oracle (needs a GB300).

pa_decode_no_alloc serves callers that cannot allocate device memory (for
instance code running inside a host application whose own allocator owns
all device memory, or a decode loop that must not call cudaMalloc/cudaFree
because they can synchronise the device): it keeps the split-KV scratch in
a built-in 40 MiB device array instead of a caller-provided workspace.

The tests call it through the C ABI several times in a row on inputs that
need that scratch, on both schedules:
  * fixed partitions (partition_size 512): output within the attention
    tolerance of pa_decode's, two calls with different queries;
  * the balanced schedule with the decode kernel merging the cut segments
    itself (the path whose arrival counters live in the shared array):
    three calls, each bit-identical to pa_decode on the same inputs (same
    kernels, same schedule) and within 2e-3 of the oracle, with the device
    error word clear after each.
The file is named to be collected last."""
import numpy as np
import pytest
import torch

import workloads as W
import paged_kv_cache_154_gb300 as pa
from gpu_harness import check_out, run_both
from paged_kv_cache_154_gb300.engine import PagedKVCache

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def built():
    from paged_kv_cache_154_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(scope="module")
def state(built):
    wl = W.simple("no_alloc", 4242, [600, 1500, 40, 1030], [1, 2, 1, 3], 32, 8, 128, "bf16")
    cache = PagedKVCache(wl.num_blocks, wl.num_kv_heads, wl.head_dim, wl.kv_dtype,
                         free_order=wl.free_order)
    names = {}
    for ops in wl.phases:
        cache.run_phase(ops, names)
    si = cache.prepare_step(wl.step, names, wl.q, torch.float32, 512)
    cache.step(si, wl.scale, 512)              # appends the step's tokens, then attends
    torch.cuda.synchronize()
    assert si.workspace is not None            # these inputs need split-KV scratch
    return wl, cache, si


def _pair(wl, cache, si, q):
    ref = torch.empty_like(si.out)
    got = torch.full_like(si.out, float("nan"))
    args = (cache.k, cache.v, si.block_tables, si.context_lens, si.max_context_len, wl.scale,
            si.query_start_loc, si.max_q_len, cache.num_blocks)
    pa.decode(ref, q, *args, partition_size=512, workspace=si.workspace)
    pa.decode_no_alloc(got, q, *args, partition_size=512)
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    return ref, got


def test_no_alloc_matches_decode_on_two_calls_in_a_row(state):
    wl, cache, si = state
    q2 = (si.q.float() * -0.5).to(si.q.dtype)          # a different query for the second call
    for q in (si.q, q2):
        ref, got = _pair(wl, cache, si, q)
        assert torch.isfinite(got).all()
        err = (got.double() - ref.double()).abs().max().item()
        assert err <= TOL, err


def test_no_alloc_balanced_in_kernel_merge_three_calls(built):
    """The balanced schedule on a call whose block bound (3 sequences x 8 KV
    heads x 750 blocks = 18,000) is at least 8 blocks per worker for any
    worker count (at most 2,048), so the decode kernel merges its cut
    segments itself through the arrival counters in the built-in array;
    the 12,000-token sequence is cut into more than 8 pieces, so its merge
    takes two levels."""
    wl = W.simple("no_alloc_balanced", 4343, [12000, 5000, 2000], [1, 1, 1], 32, 8, 128, "bf16")
    ref, cache, si, out = run_both(wl)               # pa_decode, balanced, vs the oracle
    check_out(ref, out, "bf16")
    need = pa.decode_workspace_size(3, 3, 32, 8, 128, 1, si.max_context_len, 0)
    assert 0 < need <= pa.NO_ALLOC_WORKSPACE_BYTES
    for call in range(3):
        got = torch.full_like(si.out, float("nan"))
        pa.decode_no_alloc(got, si.q, cache.k, cache.v, si.block_tables, si.context_lens,
                           si.max_context_len, wl.scale, None, 1, cache.num_blocks)
        torch.cuda.synchronize()
        assert pa.device_error() == 0, f"call {call}"
        assert torch.equal(got, out), f"call {call}: differs from pa_decode"
        check_out(ref, got, "bf16")


def test_no_alloc_rejects_workspace_beyond_its_maximum(state):
    wl, cache, si = state
    big = pa.decode_workspace_size(si.context_lens.shape[0], si.q.shape[0], wl.num_heads,
                                   wl.num_kv_heads, wl.head_dim, si.max_q_len, 1 << 17, 16)
    assert big > pa.NO_ALLOC_WORKSPACE_BYTES
    with pytest.raises(pa.PAError) as e:
        pa.decode_no_alloc(si.out, si.q, cache.k, cache.v, si.block_tables, si.context_lens,
                           1 << 17, wl.scale, si.query_start_loc, si.max_q_len,
                           cache.num_blocks, partition_size=16)
    assert e.value.status == 2 and str(pa.NO_ALLOC_WORKSPACE_BYTES) in str(e.value)

"""Runs a workload through the CUDA path and through the oracle, and
compares them: slots, copy pairs and block tables bit for bit, the whole
cache (canary blocks included) bit for bit, attention within tolerance."""
import os

import numpy as np
import torch

import oracle
import workloads as W
import paged_kv_cache_154_gb300 as pa
from paged_kv_cache_154_gb300.engine import PagedKVCache

TOL = {"f16": 2e-3, "bf16": 2e-3, "int8": 1e-2, "fp8": 2e-3}   # max abs error on attention outputs
# Regression guards, far below the tolerances: the kernels' errors on these
# inputs are about 1e-6 (16-bit), 1e-4 (FP8) and 2e-4 (INT8); a guard about
# 10x above that catches a kernel that got worse, or a dropped key block,
# long before the tolerance would. Scaled by the largest |output| where that
# exceeds 1 (inputs with a wide value range).
GUARD = {"f16": 1e-4, "bf16": 1e-4, "int8": 2e-3, "fp8": 5e-4}
THREADS = os.cpu_count() or 1


def half_ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Half a unit in the last place of |x| in `dtype` (rounding of a stored output)."""
    mant = {torch.bfloat16: 8, torch.float16: 11, torch.float32: 24}[dtype]
    ax = np.maximum(np.abs(x), 1e-30)
    return np.exp2(np.floor(np.log2(ax)) - mant)


def run_both(wl, partition_size=0, out_dtype=torch.float32, oracle_run=None,
             shared_prefix=False):
    ref = oracle_run or oracle.run(wl, threads=THREADS, canary_blocks=W.CANARY_BLOCKS,
                                   canary_byte=W.CANARY_BYTE)
    cache = PagedKVCache(wl.num_blocks, wl.num_kv_heads, wl.head_dim, wl.kv_dtype,
                         free_order=wl.free_order, canary_blocks=W.CANARY_BLOCKS,
                         canary_byte=W.CANARY_BYTE, head_scales=wl.head_scales)
    names = {}
    for ops, oslots, opairs in zip(wl.phases, ref.phase_slots, ref.phase_pairs):
        slots, pairs = cache.run_phase(ops, names)
        assert np.array_equal(slots, oslots)
        assert pairs == [tuple(p) for p in opairs]
    si = cache.prepare_step(wl.step, names, wl.q, out_dtype, partition_size,
                            shared_prefix=shared_prefix)
    assert np.array_equal(si.slots.cpu().numpy(), ref.step_slots)
    got_pairs = [] if si.pairs is None else [tuple(p) for p in si.pairs.cpu().tolist()]
    assert got_pairs == [tuple(p) for p in ref.step_pairs]
    assert np.array_equal(si.block_tables.cpu().numpy(), ref.block_tables)
    assert np.array_equal(si.context_lens.cpu().numpy(), ref.context_lens)
    out = cache.step(si, wl.scale, partition_size)
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    return ref, cache, si, out


def check_cache_bits(ref, cache):
    for dev, host in zip(cache.arrays(), ref.cache.arrays()):
        d = dev.contiguous().view(torch.uint8).cpu().numpy().reshape(-1)
        h = np.ascontiguousarray(host).view(np.uint8).reshape(-1)
        if not np.array_equal(d, h):
            bad = np.flatnonzero(d != h)
            raise AssertionError(f"cache differs at {bad.size} bytes, first at byte {bad[0]}")


def check_out(ref, out, kv_dtype, out_dtype=torch.float32, guard=True):
    got = out.double().cpu().numpy()
    err = np.abs(got - ref.out)
    tol = TOL[kv_dtype]
    if out_dtype != torch.float32:
        bound = tol + half_ulp(ref.out, out_dtype)
        assert (err <= bound).all(), f"max excess {(err - bound).max():.3e}"
    else:
        assert err.max() <= tol, f"max abs error {err.max():.3e} > {tol}"
        if guard:
            g = GUARD[kv_dtype] * max(1.0, float(np.abs(ref.out).max()))
            assert err.max() <= g, f"max abs error {err.max():.3e} above the regression guard {g:.1e}"
    return float(err.max())

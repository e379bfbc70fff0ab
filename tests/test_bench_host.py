"""Host-side logic of bench.py (no GPU): the kernels a step launches, the
kernel the roofline names, and the rule that a profile's recorded DRAM
traffic is reported only for the workload and kernel source it was captured
on."""
import numpy as np
import os
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _si(max_q_len=1, max_context_len=4096, pairs=None, shared=None, n_seqs=8, n_q=None):
    return SimpleNamespace(max_q_len=max_q_len, max_context_len=max_context_len, pairs=pairs,
                           shared=shared, context_lens=np.zeros(n_seqs),
                           q=np.zeros((n_seqs if n_q is None else n_q, 1, 1)))


def _wl(kv="bf16", H=32, Hkv=8, d=128):
    return SimpleNamespace(kv_dtype=kv, num_heads=H, num_kv_heads=Hkv, head_dim=d)


@pytest.mark.parametrize("kv, group, qlen, expect", [
    ("bf16", 4, 1, 2),      # append + decode that merges its own cut segments
    ("f16", 8, 2, 2),       # 16 rows per KV head: still the per-warp kernel
    ("bf16", 8, 3, 3),      # 24 rows: 64-row kernel + segment reduce
    ("int8", 4, 1, 3),      # INT8 decode + segment reduce
    ("fp8", 4, 1, 3),       # FP8 decode + segment reduce
])
def test_launches_per_balanced_step(kv, group, qlen, expect):
    assert bench.launches_per_step(_si(max_q_len=qlen), 0, False, kv, group) == expect


def test_launches_with_copies_partitions_prefill_and_shared_prefix():
    si = _si(pairs=object())
    assert bench.launches_per_step(si, 0, False, "bf16", 4) == 3              # + copy_blocks
    assert bench.launches_per_step(_si(max_context_len=4096), 512, False, "bf16", 4) == 3
    assert bench.launches_per_step(_si(max_context_len=400), 512, False, "bf16", 4) == 2
    assert bench.launches_per_step(_si(), 0, True, "bf16", 4) == 3            # order + prefill
    # best-of-5 shape: 5 forks x 8 q heads per KV head in the prefix phase
    # (4,096-token prefixes: split-key tensor-core kernel + chunk reduce;
    # short prefixes: 64-row kernel + reduce), 8 rows in the suffix phase
    # (decode + reduce, on the second stream); prep and merge
    sp = SimpleNamespace(max_group_q_len=5, prefix_len_host=np.array([4096] * 8))
    assert bench.prefix_tc_runs("bf16", _si(shared=sp), 8)
    assert bench.launches_per_step(_si(shared=sp), 0, False, "bf16", 8) == 1 + 2 + 2 + 2
    short = SimpleNamespace(max_group_q_len=5, prefix_len_host=np.array([512] * 8))
    assert not bench.prefix_tc_runs("bf16", _si(shared=short), 8)
    assert bench.launches_per_step(_si(shared=short), 0, False, "bf16", 8) == 1 + 2 + 2 + 2
    assert not bench.prefix_tc_runs("bf16", _si(shared=SimpleNamespace(
        max_group_q_len=1, prefix_len_host=np.array([4096]))), 8)     # 8 rows: per-warp kernel


def test_roofline_kernel_names_what_runs():
    assert "in-kernel" in bench.roofline_kernel(_wl(), _si(), 0, False)
    assert "rows_kernel + segment_reduce" in bench.roofline_kernel(_wl(), _si(max_q_len=5), 0,
                                                                   False)
    assert "int8" in bench.roofline_kernel(_wl("int8"), _si(), 0, False)
    # INT8 with 64 rows per KV head on average: the tensor-core kernel (MQA,
    # 8 sequences with 16 query tokens); 48 on average: the per-warp kernel
    mqa = _wl("int8", H=32, Hkv=1)
    assert "int8_tc" in bench.roofline_kernel(mqa, _si(max_q_len=5, n_q=16), 0, False)
    assert "int8_kernel" in bench.roofline_kernel(mqa, _si(max_q_len=5, n_q=12), 0, False)
    assert "fp8" in bench.roofline_kernel(_wl("fp8"), _si(), 0, False)
    assert "split_kv_reduce" in bench.roofline_kernel(_wl(), _si(), 512, False)
    assert "tcgen05" in bench.roofline_kernel(_wl(), _si(), 0, True)
    sp = SimpleNamespace(max_group_q_len=5, prefix_len_host=np.array([4096] * 8))
    name = bench.roofline_kernel(_wl(H=64), _si(shared=sp), 0, False)
    assert "split-key" in name and "second stream" in name


def test_recorded_traffic_only_for_the_profiled_workload():
    import re
    for key, (fname, _) in bench.PROFILES.items():
        path = os.path.join(ROOT, "profiles", fname)
        if not os.path.exists(path):
            assert bench.recorded_traffic(key) is None
            continue
        text = open(path).read()
        assert re.search(r"^workload:\s*" + re.escape(key) + r"\s*$", text, re.M), key
        fresh = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text).group(1) == \
            bench.kernel_digest(key)
        t = bench.recorded_traffic(key)
        # reported exactly when the summary was taken on the current source
        assert (t is not None and t > 0) == fresh, key
    assert bench.recorded_traffic("tiny") is None


def test_percentile():
    xs = list(range(1, 101))
    assert bench.percentile(xs, 50) == pytest.approx(50.5)
    assert bench.percentile(xs, 95) == pytest.approx(95.05)
    assert bench.percentile([3.0], 95) == 3.0


def test_every_config_run_names_a_workload_and_a_profile():
    import workloads as W
    for name, workload, shared in bench.CONFIG_RUNS:
        assert workload in W.NAMED
        assert bench.profile_key(workload, shared) in bench.PROFILES

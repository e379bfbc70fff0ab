#!/usr/bin/env python3
"""Benchmark of one paged decode step (copy-on-write block copies, KV append,
paged decode attention, split-KV reduce) through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama3_8b|tiny|llama2_70b_best_of_5|long_context]

Prints one JSON line. `value` is KV GB/s: the algorithmic bytes of a step
(K and V read by attention + q read + output written + the appended K/V
rows written) over the device time of the step, inputs resident in HBM, L2
flushed between steps (each step timed alone with CUDA events). Sequences
are independent, so N ranks each run their own replica of the batch
(weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attn KV GB/s (% of GB300 HBM peak); seq-steps/s at 1 GPU"
# Committed ncu summary per profiled workload: the summary file and the
# sources whose digest it records (traffic is reported only while they match).
_DEC16 = ("paged_decode.cu", "balanced.cuh", "ptx.cuh")
PROFILES = {
    "llama3_8b": ("paged_decode_llama3_8b.md", _DEC16),
    "llama2_70b_best_of_5": ("paged_decode_llama2_70b_best_of_5.md", _DEC16),
    "llama2_70b_best_of_5+read_once": ("shared_prefix_llama2_70b_best_of_5.md",
                                       _DEC16 + ("shared_prefix.cu", "paged_prefill_tc.cu",
                                                 "tcgen05.cuh")),
    "long_context": ("paged_decode_long_context.md", _DEC16),
    "mixed_int8": ("paged_decode_int8_mixed.md", ("paged_decode_int8.cu", "balanced.cuh",
                                                  "ptx.cuh")),
    "mqa_int8_verify": ("paged_decode_int8_tc_verify.md", ("paged_decode_int8_tc.cu", "balanced.cuh",
                                                          "ptx.cuh", "tcgen05.cuh")),
    "llama3_8b_fp8": ("paged_decode_fp8_llama3_8b.md", ("paged_decode_fp8.cu", "balanced.cuh",
                                                        "ptx.cuh")),
    "paged_prefill": ("paged_prefill_tc_llama3_8b_chunked.md",
                      ("paged_prefill_tc.cu", "tcgen05.cuh", "ptx.cuh")),
}
# The configurations timed beside the headline in a default run: (entry,
# workload, read-once shared prefixes).
CONFIG_RUNS = (
    ("llama2_70b_best_of_5", "llama2_70b_best_of_5", False),
    ("llama2_70b_best_of_5_read_once", "llama2_70b_best_of_5", True),
    ("long_context", "long_context", False),
    ("mixed_int8", "mixed_int8", False),
    ("llama3_8b_fp8", "llama3_8b_fp8", False),
    ("paged_prefill", "paged_prefill", False),
)


def profile_key(workload: str, shared_prefix: bool = False) -> str:
    return workload + ("+read_once" if shared_prefix else "")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None,
                    help="one workload alone (default: llama3_8b as the headline, with every "
                         "other configuration timed beside it under `configs`)")
    ap.add_argument("--no-configs", action="store_true",
                    help="time the headline workload only")
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="read-once decode: fork groups read their shared blocks once")
    ap.add_argument("--prefix-trace", action="store_true",
                    help="host prefix-cache trace: reuse and allocator throughput (no GPU)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_workload(name: str, rank: int):
    """This rank's shard: the named workload drawn with the rank's seed, so N
    ranks process N independent batches (weak scaling, no data exchange)."""
    import workloads as W
    return W.NAMED[name](shard=rank)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's time (the job finishes when the last rank does)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def step_bytes(wl, out_bytes_per_elem=4):
    """Algorithmic bytes of one step: every sequence's K and V for all its
    tokens (the attention must read them), q, the output, and the appended
    rows (written once)."""
    kv_elem = 1 if wl.kv_dtype in ("int8", "fp8") else 2
    per_tok = 2 * wl.num_kv_heads * wl.head_dim * kv_elem
    if wl.kv_dtype == "int8":
        per_tok += 2 * wl.num_kv_heads * 5          # fp32 scale + int8 zero point, K and V
    kv_read = sum(wl.context_lens) * per_tok
    nq = sum(wl.q_lens)
    q_b = nq * wl.num_heads * wl.head_dim * 2
    out_b = nq * wl.num_heads * wl.head_dim * out_bytes_per_elem
    appended = nq * per_tok
    return {"kv_read": kv_read, "q": q_b, "out": out_b, "append_write": appended,
            "decode": kv_read + q_b + out_b, "step": kv_read + q_b + out_b + appended}


def kernel_digest(key: str = "llama3_8b"):
    h = hashlib.sha256()
    for f in PROFILES[key][1]:
        with open(os.path.join(ROOT, "paged_kv_cache_154_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(key: str):
    """DRAM bytes (read + write) of one attention call from the committed ncu
    summary of this workload, if it was taken on the current kernel source;
    else None."""
    if key not in PROFILES:
        return None
    try:
        text = open(os.path.join(ROOT, "profiles", PROFILES[key][0])).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_call:\s*([0-9.eE+]+)", text)
    m_w = re.search(r"^workload:\s*(\S+)", text, re.M)
    if not m_sha or not m_b or m_sha.group(1) != kernel_digest(key):
        return None
    if not m_w or m_w.group(1) != key:
        return None
    return float(m_b.group(1))


def measured_peak(key: str = "hbm_gbs"):
    fallback = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)[key]), "measured"
    except Exception:
        return fallback[key], "fallback"


def attention_flops(wl) -> int:
    """Multiply-adds of the causal attention, x2: each query row (query i of
    a run of r at position L - r + i, every q head) against its L - r + i + 1
    keys, for Q K^T and for P V."""
    tot = 0
    for L, r in zip(wl.context_lens, wl.q_lens):
        tot += r * (L - r + 1) + r * (r - 1) // 2
    return 4 * wl.head_dim * wl.num_heads * tot


def is_prefill(wl) -> bool:
    return max(wl.q_lens) > 16


class ClockSampler:
    """nvidia-smi sampled every 50 ms in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.samples = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                self.samples.append({"sm": float(parts[1]), "max": float(parts[2]),
                                     "hw": parts[4], "hw_thermal": parts[5],
                                     "sw_thermal": parts[6], "sw_power": parts[7]})
            except ValueError:
                pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sms = [s["sm"] for s in self.samples]
        reasons = set()
        for s in self.samples:
            for k, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                            ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if s[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(s["max"] for s in self.samples),
                "reasons": sorted(reasons), "samples": len(sms)}


def build_state(wl, device, partition_size, shared_prefix=False):
    import torch
    from paged_kv_cache_154_gb300.engine import PagedKVCache
    cache = PagedKVCache(wl.num_blocks, wl.num_kv_heads, wl.head_dim, wl.kv_dtype,
                         device=device, free_order=wl.free_order, head_scales=wl.head_scales)
    names = {}
    for ops in wl.phases:
        cache.run_phase(ops, names)
    si = cache.prepare_step(wl.step, names, wl.q, torch.float32, partition_size,
                            shared_prefix=shared_prefix)
    torch.cuda.synchronize()
    return cache, si, names


def unique_kv_bytes(wl, group_start, prefix_len):
    """KV bytes read-once decode must read: each group's shared prefix once,
    every sequence's tokens after it once."""
    per_tok = 2 * wl.num_kv_heads * wl.head_dim * (1 if wl.kv_dtype in ("int8", "fp8") else 2)
    toks = 0
    for g in range(len(prefix_len)):
        toks += int(prefix_len[g])
        for s in range(int(group_start[g]), int(group_start[g + 1])):
            toks += wl.context_lens[s] - int(prefix_len[g])
    return toks * per_tok


def launches_per_step(si, partition_size, prefill_tc=False, kv_dtype="bf16", group=1):
    """Kernels of one step. A balanced decode over a 16-bit cache with at most
    16 query rows per KV head merges its cut segments itself; every other
    balanced decode launches the segment reduce after it."""
    def decode_launches(rows, balanced=True, long_enough=True):
        if not balanced:
            return 1 + (1 if long_enough else 0)        # decode (+ partition reduce)
        fused = kv_dtype in ("f16", "bf16") and rows <= 16
        return 1 if fused else 2                        # decode (+ segment reduce)

    n = 1                                               # append
    if si.pairs is not None:
        n += 1                                          # copy_blocks
    if si.shared is not None:
        # prep, the prefix phase (on the tensor cores: split-key kernel and
        # chunk reduce), the suffix phase (always with its reduce kernel),
        # the merge of the two
        prefix = (2 if prefix_tc_runs(kv_dtype, si, group)
                  else decode_launches(group * si.shared.max_group_q_len))
        return n + 2 + prefix + 2
    if prefill_tc:
        return n + 2                                    # task order, tensor-core prefill
    return n + decode_launches(group * si.max_q_len, partition_size == 0,
                               si.max_context_len > partition_size)


def prefix_tc_runs(kv_dtype, si, group, head_dim=128) -> bool:
    """Does the read-once prefix phase run on the tensor-core kernel (16-bit
    cache, head_dim 128, 17-64 rows per group and KV head, prefixes of at
    least 1,024 tokens)?"""
    rows = group * si.shared.max_group_q_len
    return (kv_dtype in ("f16", "bf16") and head_dim == 128 and 16 < rows <= 64
            and int(max(si.shared.prefix_len_host)) >= 1024)


def int8_tc_runs(wl, si) -> bool:
    """Whether an INT8 call takes the tensor-core kernel: head_dim 128, more
    than 16 query rows per KV head at most and at least 64 on average (the
    library's own rule)."""
    G = wl.num_heads // wl.num_kv_heads
    n_seqs = si.context_lens.shape[0]
    n_q = si.q.shape[0]
    return (wl.head_dim == 128 and G * si.max_q_len > 16 and G * n_q >= 64 * n_seqs
            and n_seqs <= 1536)


def roofline_kernel(wl, si, partition_size, prefill_tc):
    """The kernels the timed attention call launches."""
    G = wl.num_heads // wl.num_kv_heads

    def balanced16(rows):
        return ("paged_decode_balanced_kernel (cut segments merged in-kernel)" if rows <= 16
                else "paged_decode_rows_kernel + segment_reduce_kernel")

    if prefill_tc:
        return ("pa_decode (paged_prefill_tc_kernel: Q K^T and P V on the tcgen05 tensor "
                "cores, accumulators in TMEM)")
    if si.shared is not None:
        prefix = ("paged_prefill_tc_kernel in split-key mode (tcgen05, TMEM) + "
                  "prefix_chunk_reduce_kernel" if prefix_tc_runs(wl.kv_dtype, si, G, wl.head_dim)
                  else balanced16(G * si.shared.max_group_q_len))
        suffix = ("paged_decode_balanced_kernel" if G * si.max_q_len <= 16
                  else "paged_decode_rows_kernel") + " + segment_reduce_rows_kernel"
        return (f"pa_decode_shared_prefix (prefix_prep_kernel, {prefix} for the prefixes, "
                f"{suffix} for the suffixes on a second stream beside them, "
                f"prefix_merge_kernel)")
    if wl.kv_dtype == "int8":
        return ("pa_decode (paged_decode_int8_tc_kernel: tokens in M on the tcgen05 tensor cores, "
                "+ segment_reduce_kernel)" if int8_tc_runs(wl, si) else
                "pa_decode (paged_decode_int8_kernel + segment_reduce_kernel)")
    if wl.kv_dtype == "fp8":
        return "pa_decode (paged_decode_fp8_kernel + segment_reduce_kernel)"
    if partition_size == 0:
        return f"pa_decode ({balanced16(G * si.max_q_len)})"
    return "pa_decode (paged_decode_kernel + split_kv_reduce_kernel)"


def percentile(xs, q):
    """The q-th percentile (0..100) of xs, linear between order statistics."""
    ys = sorted(xs)
    if len(ys) == 1:
        return ys[0]
    x = (len(ys) - 1) * q / 100.0
    i = int(x)
    j = min(i + 1, len(ys) - 1)
    return ys[i] + (ys[j] - ys[i]) * (x - i)


def time_workload(wl, device, steps, warmup, partition_size=0, shared_prefix=False, world=1,
                  local=0, keep_state=False):
    """Times `steps` steps of one workload on this rank: each step the cache
    writes (copy-on-write copies, append) and the attention call, replayed
    from two CUDA graphs, timed with CUDA events on the launching stream, L2
    flushed before each step outside the timed window. Returns the timings
    and, with keep_state, the device state for the end-to-end leg."""
    import torch
    import paged_kv_cache_154_gb300 as pa
    if shared_prefix and partition_size:
        raise SystemExit("--shared-prefix uses the balanced schedule (partition size 0)")
    cache, si, names = build_state(wl, device, partition_size, shared_prefix)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(2 * max(l2, 64 << 20), dtype=torch.uint8, device=device)
    clean = torch.ones(2 * max(l2, 64 << 20) // 4, dtype=torch.float32, device=device)

    def flush_l2(k):
        # write a buffer twice the L2 (evicts the previous step), then read another
        # one, so the dirty lines are written back here, outside the timed window
        flush.fill_(k & 0xFF)
        clean.sum()

    # the step as two CUDA graphs (cache writes; attention), replayed back to back
    g_write = cache.capture(cache.write_step, si)
    g_attend = cache.capture(cache.attend_step, si, wl.scale, partition_size)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(max(3, warmup)):
        g_write.replay()
        g_attend.replay()
    torch.cuda.synchronize()
    assert pa.device_error() == 0
    K = steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local)
    time.sleep(0.15)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for k in range(K):
        flush_l2(k)
        ev[k][0].record(stream)
        g_write.replay()
        ev[k][1].record(stream)
        g_attend.replay()
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall1 = time.perf_counter()
    time.sleep(0.1)
    sampler.stop()
    assert pa.device_error() == 0
    res = {"step_ms": [ev[k][0].elapsed_time(ev[k][2]) for k in range(K)],
           "dec_ms": [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)],
           "clocks": sampler.summary(), "wall_s": wall1 - wall0,
           "si_info": {"pairs": si.pairs is not None, "max_q_len": si.max_q_len,
                       "max_context_len": si.max_context_len,
                       "shared": (None if si.shared is None else
                                  (si.shared.group_start_host, si.shared.prefix_len_host,
                                   si.shared.max_group_q_len))}}
    res["launches"] = launches_per_step(si, partition_size, prefill_tc_runs(wl, partition_size,
                                                                            si),
                                        wl.kv_dtype, wl.num_heads // wl.num_kv_heads)
    res["kernel"] = roofline_kernel(wl, si, partition_size,
                                    prefill_tc_runs(wl, partition_size, si))
    del g_write, g_attend, flush, clean
    if keep_state:
        res["state"] = (cache, si, names)
    else:
        del cache, si
        torch.cuda.empty_cache()
    return res


def prefill_tc_runs(wl, partition_size, si) -> bool:
    """Does the library send this step's attention to the tensor-core prefill
    kernel? (long query runs over a 16-bit cache with head_dim 128)."""
    return (is_prefill(wl) and wl.kv_dtype in ("bf16", "f16") and wl.head_dim == 128
            and partition_size == 0 and si.shared is None)


def roofline_entry(wl, res, key, shared_prefix=False):
    """The attention call's roofline: algorithmic bytes (or, for prefill,
    flops) per call over its mean event time, against the measured peak."""
    nbytes = step_bytes(wl)
    sh = res["si_info"]["shared"]
    if sh is not None:
        nbytes["kv_read_unique"] = unique_kv_bytes(wl, sh[0], sh[1])
        nbytes["decode_unique"] = nbytes["kv_read_unique"] + nbytes["q"] + nbytes["out"]
    dec = res["dec_ms"]
    dec_avg_s = statistics.mean(dec) / 1e3
    if is_prefill(wl):
        units = attention_flops(wl)
        peak, kind = measured_peak("bf16_tflops")
        achieved, unit, bound = units / dec_avg_s / 1e12, "TFLOP/s", "tensor"
        ukey = "algorithmic_flops_per_launch"
    else:
        # the method's own algorithmic bytes: read-once decode reads shared blocks once
        units = nbytes.get("decode_unique", nbytes["decode"])
        peak, kind = measured_peak("hbm_gbs")
        achieved, unit, bound = units / dec_avg_s / 1e9, "GB/s", "hbm"
        ukey = "algorithmic_bytes_per_launch"
    roof = {"kernel": res["kernel"], "bound": bound, "achieved": round(achieved, 1),
            "peak": peak, "peak_kind": kind, "unit": unit, "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(key), ukey: units,
            "decode_ms_avg": round(dec_avg_s * 1e3, 5),
            "decode_ms_p50": round(statistics.median(dec), 5),
            "decode_ms_p95": round(percentile(dec, 95), 5)}
    if sh is not None:
        roof["logical_bytes_per_launch"] = nbytes["decode"]
        roof["logical_gbs"] = round(nbytes["decode"] / dec_avg_s / 1e9, 1)
    return roof, nbytes


def config_entry(name, workload, shared_prefix, device, steps, warmup):
    """One configuration's timings as a `configs` entry of the bench line."""
    import workloads as W
    wl = W.NAMED[workload]()
    res = time_workload(wl, device, steps, warmup, 0, shared_prefix)
    key = profile_key(workload, shared_prefix)
    roof, nbytes = roofline_entry(wl, res, key, shared_prefix)
    tot_s = sum(res["step_ms"]) / 1e3
    return {"workload": workload, "read_once_shared_prefix": shared_prefix,
            "dtype": wl.kv_dtype, "steps": steps,
            "value": round(steps * nbytes["step"] / tot_s / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(1e3 * tot_s / steps, 5),
            "seq_steps_per_s": round(steps * wl.num_seqs / tot_s, 1),
            "num_seqs": wl.num_seqs, "heads": [wl.num_heads, wl.num_kv_heads],
            "head_dim": wl.head_dim, "context_tokens": sum(wl.context_lens),
            "query_tokens": sum(wl.q_lens), "bytes_per_step": nbytes, "roofline": roof,
            "gpu_launches_per_step": res["launches"], "clocks": res["clocks"]}


def run_ours(args, rank, world, local):
    import torch

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    workload = args.workload or "llama3_8b"
    wl = rank_workload(workload, rank)
    res = time_workload(wl, device, args.steps, args.warmup, args.partition_size,
                        args.shared_prefix, world, local, keep_state=True)
    nbytes = step_bytes(wl)
    K = args.steps
    tot_ms = max_over_ranks(sum(res["step_ms"]), world, device)
    job_bytes = sum_over_ranks(float(nbytes["step"]), world, device)
    job_seqs = sum_over_ranks(float(wl.num_seqs), world, device)

    # end to end through the public API: host pool, pinned host buffers, C-ABI calls
    cache, si, names = res.pop("state")
    e2e = None
    if not args.shared_prefix and args.partition_size == 0:
        e2e = measure_e2e(wl, cache, si, names, steps=min(K, 50))
    del cache, si
    torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    key = profile_key(workload, args.shared_prefix)
    roof, nbytes = roofline_entry(wl, res, key, args.shared_prefix)
    hbm_peak, _ = measured_peak()
    value = K * job_bytes / (tot_ms / 1e3) / 1e9
    seq_steps = K * job_seqs / (tot_ms / 1e3)
    si_info = res["si_info"]
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(tot_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.kv_dtype,
        "data": "synthetic (seeded N(0,1) K/V/q, seeded lengths and block placement)",
        "config": {"workload": wl.name, "num_seqs": wl.num_seqs, "num_heads": wl.num_heads,
                   "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                   "block_size": 16, "context_tokens": sum(wl.context_lens),
                   "schedule": ("balanced, read-once shared prefixes "
                                f"({len(si_info['shared'][1])} fork groups)"
                                if si_info["shared"] is not None else
                                "balanced" if args.partition_size == 0
                                else f"partitions of {args.partition_size}"),
                   "l2": "flushed between steps (2x L2 write, then a 2x L2 read so no dirty "
                         "line is left), each step timed alone",
                   "launch": "CUDA graphs (cache writes; attention) replayed per step",
                   "bytes_per_step": nbytes,
                   "parallelism": (f"{world} ranks, one shard of independent sequences each"
                                   if world > 1 else "1 GPU")},
        "seq_steps_per_s": round(seq_steps, 1),
        "pct_of_hbm_peak": round(100 * value / hbm_peak, 2),
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": res["launches"] * K,
        "clocks": res["clocks"],
        "wall_s_timed": round(res["wall_s"], 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=12.0)
    # the other configurations, each timed on its own (default run only)
    if world == 1 and args.workload is None and not args.no_configs:
        line["configs"] = {}
        for name, w, sp in CONFIG_RUNS:
            line["configs"][name] = config_entry(name, w, sp, device, max(50, K), args.warmup)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_e2e(wl, cache, si, names, steps):
    """The same metric through the public API, as a user's decode loop runs
    it, every step: the host pool reserves the step's new slots in one call
    (pa_seq_append_slots_batch; the copy-on-write pairs come back) and writes
    the block tables and lengths; those, the step's q and new K/V rows are
    packed in one pinned host buffer and copied to the device in one copy;
    pa_copy_blocks (when there are pairs), pa_append_kv and pa_decode run;
    the output is copied back to pinned host memory and the stream
    synchronised. The sequences grow by their query run each step, and each
    step's bytes are counted from its own lengths."""
    import numpy as np
    import torch
    import paged_kv_cache_154_gb300 as pa
    dev = si.q.device
    seqs = [names[op.seq] for op in wl.step]
    q_lens = [int(op.k.shape[0]) for op in wl.step]
    seqs_np = np.asarray(seqs, np.int32)
    q_lens_np = np.asarray(q_lens, np.int32)
    r_max = max(q_lens)
    T = sum(q_lens)
    warm = 3
    cap_blocks = si.block_tables.shape[1] + ((warm + steps) * r_max + 15) // 16 + 1
    max_len_final = si.max_context_len + (warm + steps) * r_max
    ws_bytes = pa.decode_workspace_size(len(seqs), T, wl.num_heads, wl.num_kv_heads,
                                        wl.head_dim, r_max, max_len_final, 0)
    ws = pa.zeroed_workspace(ws_bytes, dev)
    # one pinned host staging buffer and one device buffer holding every
    # input of a step, as typed views at 256-byte offsets
    parts = [("slots", (T,), torch.int64), ("bt", (len(seqs), cap_blocks), torch.int32),
             ("cl", (len(seqs),), torch.int32), ("q", tuple(si.q.shape), si.q.dtype),
             ("key", tuple(si.key.shape), si.key.dtype),
             ("value", tuple(si.value.shape), si.value.dtype)]
    offs, total = {}, 0
    for name, shape, dt in parts:
        offs[name] = total
        nb = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        total += (nb + 255) // 256 * 256
    stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, name):
        _, shape, dt = next(x for x in parts if x[0] == name)
        nb = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        return buf[offs[name]:offs[name] + nb].view(dt).view(shape)

    h = {name: view(stage_h, name) for name, _, _ in parts}
    d = {name: view(stage_d, name) for name, _, _ in parts}
    for name in ("q", "key", "value"):
        h[name].copy_(getattr(si, name).cpu())
    qsl = si.query_start_loc            # fixed: the run lengths do not change
    out_h = torch.empty(si.out.shape, dtype=si.out.dtype).pin_memory()
    out_d = torch.empty_like(si.out)
    stream = torch.cuda.current_stream()
    # the sequences grow by their query run every step: the pool must have room
    free_blocks = cache.pool.stats()[0]
    need = sum(((warm + steps) * r + 15) // 16 + 1 for r in q_lens)
    if need > free_blocks:
        return {"value": None, "unit": "GB/s",
                "note": f"pool has {free_blocks} free blocks, {warm + steps} growing steps need "
                        f"{need}: not measured for this workload"}
    kv_elem = 1 if wl.kv_dtype in ("int8", "fp8") else 2
    per_tok = 2 * wl.num_kv_heads * wl.head_dim * kv_elem + (
        2 * wl.num_kv_heads * 5 if wl.kv_dtype == "int8" else 0)
    fixed = T * wl.num_heads * wl.head_dim * (2 + 4) + T * per_tok
    slots_np = h["slots"].numpy()
    bt_np, cl_np = h["bt"].numpy(), h["cl"].numpy()
    pr_h = torch.empty((len(seqs), 2), dtype=torch.int32).pin_memory()
    pr_d = torch.empty((len(seqs), 2), dtype=torch.int32, device=dev)
    times, nbytes, h2d_last = [], 0, 0
    for k in range(warm + steps):
        t0 = time.perf_counter()
        _, pairs = cache.pool.seq_append_slots_batch(seqs_np, q_lens_np, slots_out=slots_np)
        bt, cl = cache.pool.block_tables(seqs_np, cap_blocks)
        bt_np[:] = bt
        cl_np[:] = cl
        stage_d.copy_(stage_h, non_blocking=True)
        h2d = total
        if len(pairs):
            pr_h[:len(pairs)] = torch.from_numpy(pairs)
            pr_d[:len(pairs)].copy_(pr_h[:len(pairs)], non_blocking=True)
            h2d += len(pairs) * 8
            pa.copy_blocks(cache.k, cache.v, pr_d[:len(pairs)], cache.num_blocks, cache.k_scale,
                           cache.v_scale, cache.k_zp, cache.v_zp)
        pa.append_kv(d["key"], d["value"], cache.k, cache.v, d["slots"], cache.num_blocks,
                     cache.k_scale, cache.v_scale, cache.k_zp, cache.v_zp)
        max_len = int(cl.max())
        pa.decode(out_d, d["q"], cache.k, cache.v, d["bt"], d["cl"], max_len, wl.scale, qsl,
                  si.max_q_len, cache.num_blocks, cache.k_scale, cache.v_scale, cache.k_zp,
                  cache.v_zp, 0, ws)
        out_h.copy_(out_d, non_blocking=True)
        stream.synchronize()
        if k >= warm:
            times.append(time.perf_counter() - t0)
            nbytes += int(cl.astype(np.int64).sum()) * per_tok + fixed
            h2d_last = h2d
    assert pa.device_error() == 0
    d2h = out_h.numel() * out_h.element_size()
    return {"value": round(nbytes / sum(times) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d_last), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(1e3 * statistics.mean(times), 4), "steps": len(times),
            "path": "host pool (pa_seq_append_slots_batch, pa_pool_block_tables) + one pinned "
                    "H2D copy of the step's inputs + pa_copy_blocks/pa_append_kv/pa_decode + D2H, "
                    "per step"}


def cpu_baseline(wl, budget_s=12.0, sample_seqs=None):
    """The oracle (plain C, fp64, OpenMP over (sequence, kv head)) on a
    bounded sample of the workload's sequences, same metric (GB/s of the
    attention's algorithmic bytes for the sampled sequences), with every
    host core and with one thread."""
    import oracle
    threads = os.cpu_count() or 1
    run = oracle.run(wl, decode=False)

    def timed(n, nthreads, budget):
        qsl = wl.query_start_loc[: n + 1]
        kv_elem = 1 if wl.kv_dtype in ("int8", "fp8") else 2
        nbytes = sum(2 * wl.context_lens[s] * wl.num_kv_heads * wl.head_dim * kv_elem
                     for s in range(n))
        nq = int(qsl[-1])
        nbytes += nq * wl.num_heads * wl.head_dim * (2 + 4)
        reps, t_total = 0, 0.0
        while t_total < budget and reps < 50:
            t0 = time.perf_counter()
            oracle.attend(run.q64[:nq], run.cache, run.block_tables[:n], run.context_lens[:n],
                          qsl, wl.num_heads, wl.scale, threads=nthreads)
            t_total += time.perf_counter() - t0
            reps += 1
        return reps * nbytes / t_total / 1e9, reps, t_total

    n = wl.num_seqs if sample_seqs is None else min(sample_seqs, wl.num_seqs)
    v, reps, t = timed(n, threads, budget_s)
    n1 = min(n, 4)
    v1, reps1, t1 = timed(n1, 1, budget_s / 3)
    return {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {wl.num_seqs} sequences (all heads), attention only, "
                      f"{reps} repetitions in {t:.1f} s",
            "single_thread": {"value": round(v1, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{n1} of {wl.num_seqs} sequences (all heads), "
                                        f"attention only, {reps1} repetitions in {t1:.1f} s"}}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step one bounded sample of the
    workload on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import workloads as W
    import oracle
    wl = W.NAMED[args.workload or "llama3_8b"]()
    threads = os.cpu_count() or 1
    run = oracle.run(wl, decode=False)
    # bounded sample: the first sequences whose keys add up to ~1/8 of the batch
    target = sum(wl.context_lens) / 8
    n, acc = 0, 0
    while n < wl.num_seqs and acc < target:
        acc += wl.context_lens[n]
        n += 1
    qsl = wl.query_start_loc[: n + 1]
    nq = int(qsl[-1])
    kv_elem = 1 if wl.kv_dtype in ("int8", "fp8") else 2
    nbytes = sum(2 * wl.context_lens[s] * wl.num_kv_heads * wl.head_dim * kv_elem
                 for s in range(n)) + nq * wl.num_heads * wl.head_dim * 6

    def step():
        oracle.attend(run.q64[:nq], run.cache, run.block_tables[:n], run.context_lens[:n],
                      qsl, wl.num_heads, wl.scale, threads=threads)

    for _ in range(max(3, args.warmup) if args.warmup < 3 else args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps * nbytes / dt / 1e9
    sample = f"{n} of {wl.num_seqs} sequences (all heads) per step, attention only"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * dt / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def prefix_trace(args):
    """Prefix caching on a serving-like trace (page 1 §2.4: requests that
    share a system prompt reuse its KV): 8 system prompts of 100-1500 tokens
    chosen with Zipf-like weights, 50-400 user tokens, 20-200 generated tokens,
    at most 64 requests alive (the oldest finishes first). Reports the share
    of prompt tokens served from cached blocks, the KV append bytes that saves
    for a Llama-3-8B layer (8 KV heads x 128 x bf16, K and V), and host
    requests/s of the library's pool next to the allocator model's."""
    import numpy as np
    import paged_kv_cache_154_gb300 as pa
    from oracle.allocator import BlockPool
    rng = np.random.default_rng(1540)
    prompts = [rng.integers(0, 32000, size=int(n)).tolist()
               for n in rng.integers(100, 1500, size=8)]
    w = 1.0 / np.arange(1, 9)
    w /= w.sum()
    n_req = max(200, 20 * args.steps)
    reqs = []
    for _ in range(n_req):
        p = prompts[int(rng.choice(8, p=w))]
        user = rng.integers(0, 32000, size=int(rng.integers(50, 400))).tolist()
        gen = rng.integers(0, 32000, size=int(rng.integers(20, 200))).tolist()
        reqs.append((p + user, gen))
    num_blocks = 64 * 2200 // 16

    def run(pool, create, append, free):
        pool.enable_prefix_cache(num_blocks // 4)
        live, cached, prompt = [], 0, 0
        t0 = time.perf_counter()
        for toks, gen in reqs:
            if len(live) == 64:
                free(live.pop(0))
            sid, n = create(toks)
            append(sid, toks[n:])
            append(sid, gen)
            live.append(sid)
            cached += n
            prompt += len(toks)
        return time.perf_counter() - t0, cached, prompt

    c = pa.Pool(num_blocks, 16)
    t_lib, cached, prompt = run(c, c.create_with_prefix, c.append_tokens, c.seq_free)
    m = BlockPool(num_blocks, 16)
    t_model, cached_m, _ = run(m, m.create_with_prefix, m.append_tokens, m.release)
    assert cached == cached_m
    kv_tok = 2 * 8 * 128 * 2
    line = {"metric": "prefix-cache admissions/s (host block pool, serving trace)",
            "value": round(len(reqs) / t_lib, 1), "unit": "requests/s",
            "higher_is_better": True, "data": "synthetic token trace",
            "config": {"workload": "prefix_cache_trace", "requests": len(reqs),
                       "system_prompts": 8, "max_live": 64, "pool_blocks": num_blocks},
            "prompt_tokens_cached_frac": round(cached / prompt, 4),
            "append_bytes_saved_per_request": int(cached * kv_tok / len(reqs)),
            "cpu_baseline": {"value": round(len(reqs) / t_model, 1), "unit": "requests/s",
                             "cores": 1, "kind": "oracle",
                             "sample": "the allocator model on the same trace"}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.prefix_trace:
        if rank == 0:
            prefix_trace(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()

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
# Committed ncu summary per decode kernel family: the summary file and the
# sources whose digest it records (traffic is reported only while they match).
PROFILES = {
    "16bit": ("paged_decode_llama3_8b.md", ("paged_decode.cu", "balanced.cuh", "ptx.cuh")),
    "int8": ("paged_decode_int8_mixed.md", ("paged_decode_int8.cu", "balanced.cuh", "ptx.cuh")),
    "fp8": ("paged_decode_fp8_llama3_8b.md", ("paged_decode_fp8.cu", "balanced.cuh", "ptx.cuh")),
    "prefill": ("paged_prefill_tc_llama3_8b_chunked.md",
                ("paged_prefill_tc.cu", "tcgen05.cuh", "ptx.cuh")),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b")
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


def kernel_family(kv_dtype: str) -> str:
    return kv_dtype if kv_dtype in ("int8", "fp8") else "16bit"


def kernel_digest(family: str = "16bit"):
    h = hashlib.sha256()
    for f in PROFILES[family][1]:
        with open(os.path.join(ROOT, "paged_kv_cache_154_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(family: str = "16bit", workload: str = ""):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source and on this workload; else None."""
    try:
        text = open(os.path.join(ROOT, "profiles", PROFILES[family][0])).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_w = re.search(r"^workload:\s*(\S+)", text, re.M)
    if not m_sha or not m_b or m_sha.group(1) != kernel_digest(family):
        return None
    if not m_w or m_w.group(1) != workload:
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
    return cache, si


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
        # prep, the prefix phase, the suffix phase, the merge of the two
        return (n + 2 + decode_launches(group * si.shared.max_group_q_len)
                + decode_launches(group * si.max_q_len))
    if prefill_tc:
        return n + 2                                    # task order, tensor-core prefill
    return n + decode_launches(group * si.max_q_len, partition_size == 0,
                               si.max_context_len > partition_size)


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
        return (f"pa_decode_shared_prefix (prefix_prep_kernel, "
                f"{balanced16(G * si.shared.max_group_q_len)} for the prefixes, "
                f"{balanced16(G * si.max_q_len)} for the suffixes, prefix_merge_kernel)")
    if wl.kv_dtype == "int8":
        return "pa_decode (paged_decode_int8_kernel + segment_reduce_kernel)"
    if wl.kv_dtype == "fp8":
        return "pa_decode (paged_decode_fp8_kernel + segment_reduce_kernel)"
    if partition_size == 0:
        return f"pa_decode ({balanced16(G * si.max_q_len)})"
    return "pa_decode (paged_decode_kernel + split_kv_reduce_kernel)"


def run_ours(args, rank, world, local):
    import torch
    import workloads as W
    import paged_kv_cache_154_gb300 as pa

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    wl = rank_workload(args.workload, rank)
    if args.shared_prefix and args.partition_size:
        raise SystemExit("--shared-prefix uses the balanced schedule (partition size 0)")
    cache, si = build_state(wl, device, args.partition_size, args.shared_prefix)
    nbytes = step_bytes(wl)
    if si.shared is not None:
        nbytes["kv_read_unique"] = unique_kv_bytes(wl, si.shared.group_start_host,
                                                   si.shared.prefix_len_host)
        nbytes["decode_unique"] = nbytes["kv_read_unique"] + nbytes["q"] + nbytes["out"]
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
    g_attend = cache.capture(cache.attend_step, si, wl.scale, args.partition_size)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(max(3, args.warmup)):
        g_write.replay()
        g_attend.replay()
    torch.cuda.synchronize()
    assert pa.device_error() == 0

    K = args.steps
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
    step_ms = [ev[k][0].elapsed_time(ev[k][2]) for k in range(K)]
    dec_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)]
    tot_ms = max_over_ranks(sum(step_ms), world, device)
    job_bytes = sum_over_ranks(float(nbytes["step"]), world, device)
    job_seqs = sum_over_ranks(float(wl.num_seqs), world, device)

    # end to end: host (pinned) inputs copied in, result copied out, every step
    e2e = measure_e2e(wl, cache, si, args, (g_write, g_attend), K_e2e=min(K, 50))

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peak, peak_kind = measured_peak()
    hbm_peak = peak
    dec_avg_s = statistics.mean(dec_ms) / 1e3
    # the method's own algorithmic bytes: read-once decode reads shared blocks once
    alg_bytes = nbytes.get("decode_unique", nbytes["decode"])
    achieved = alg_bytes / dec_avg_s / 1e9
    roof_unit, bound, alg_units = "GB/s", "hbm", alg_bytes
    # the library sends long query runs over a 16-bit cache with head_dim 128
    # to the tensor-core prefill kernel
    prefill_tc = (is_prefill(wl) and wl.kv_dtype in ("bf16", "f16") and wl.head_dim == 128
                  and args.partition_size == 0 and si.shared is None
                  and "PA_PREFILL_MMA_SYNC" not in os.environ)
    if is_prefill(wl):
        # long query runs: a contraction on the tensor cores, not a KV stream
        flops = attention_flops(wl)
        peak, peak_kind = measured_peak("bf16_tflops")
        achieved = flops / dec_avg_s / 1e12
        roof_unit, bound, alg_units = "TFLOP/s", "tensor", flops
    value = K * job_bytes / (tot_ms / 1e3) / 1e9
    seq_steps = K * job_seqs / (tot_ms / 1e3)
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
                                f"({len(si.shared.prefix_len_host)} fork groups)"
                                if si.shared is not None else
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
        "roofline": {"kernel": roofline_kernel(wl, si, args.partition_size, prefill_tc),
                     "bound": bound, "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": roof_unit,
                     "frac": round(achieved / peak, 4),
                     "traffic": (recorded_traffic("prefill", args.workload) if prefill_tc else
                                 recorded_traffic(kernel_family(wl.kv_dtype), args.workload)
                                 if args.partition_size == 0 and si.shared is None
                                 and not is_prefill(wl) else None),
                     ("algorithmic_flops_per_launch" if bound == "tensor"
                      else "algorithmic_bytes_per_launch"): alg_units,
                     "decode_ms_avg": round(dec_avg_s * 1e3, 5),
                     "decode_ms_p50": round(statistics.median(dec_ms), 5)},
        "e2e": e2e,
        "gpu_launches": launches_per_step(si, args.partition_size, prefill_tc, wl.kv_dtype,
                                          wl.num_heads // wl.num_kv_heads) * K,
        "clocks": sampler.summary(),
        "wall_s_timed": round(wall1 - wall0, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=12.0)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_e2e(wl, cache, si, args, graphs, K_e2e):
    """Same metric through the public API with host buffers: per step, copy
    q, the new K/V rows, the slots, block tables, lengths (and copy pairs)
    from pinned host memory, run the step, copy the output back, sync."""
    import torch
    import paged_kv_cache_154_gb300 as pa
    pairs = []                                   # (device input, pinned host copy)
    for name in ("q", "key", "value", "slots", "block_tables", "context_lens", "pairs",
                 "query_start_loc"):
        t = getattr(si, name)
        if t is not None:
            pairs.append((t, t.cpu().pin_memory()))
    if si.shared is not None:                    # the step's fork groups are inputs too
        for t in (si.shared.group_start, si.shared.prefix_len):
            pairs.append((t, t.cpu().pin_memory()))
    out_h = torch.empty(si.out.shape, dtype=si.out.dtype).pin_memory()
    h2d = sum(h.numel() * h.element_size() for _, h in pairs)
    d2h = out_h.numel() * out_h.element_size()
    stream = torch.cuda.current_stream()
    times = []
    for k in range(K_e2e + 3):
        t0 = time.perf_counter()
        for d, h in pairs:
            d.copy_(h, non_blocking=True)
        for g in graphs:
            g.replay()
        out_h.copy_(si.out, non_blocking=True)
        stream.synchronize()
        if k >= 3:
            times.append(time.perf_counter() - t0)
    nbytes = step_bytes(wl)["step"]
    return {"value": round(len(times) * nbytes / sum(times) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(1e3 * statistics.mean(times), 4), "steps": len(times)}


def cpu_baseline(wl, budget_s=12.0, sample_seqs=None):
    """The oracle (plain C, fp64, OpenMP over (sequence, kv head)) on a
    bounded sample of the workload's sequences, same metric (GB/s of the
    attention's algorithmic bytes for the sampled sequences)."""
    import numpy as np
    import oracle
    threads = os.cpu_count() or 1
    run = oracle.run(wl, decode=False)
    n = wl.num_seqs if sample_seqs is None else min(sample_seqs, wl.num_seqs)
    qsl = wl.query_start_loc[: n + 1]
    nbytes = 0
    kv_elem = 1 if wl.kv_dtype in ("int8", "fp8") else 2
    for s in range(n):
        nbytes += 2 * wl.context_lens[s] * wl.num_kv_heads * wl.head_dim * kv_elem
    nq = int(qsl[-1])
    nbytes += nq * wl.num_heads * wl.head_dim * (2 + 4)
    reps, t_total = 0, 0.0
    while t_total < budget_s and reps < 50:
        t0 = time.perf_counter()
        oracle.attend(run.q64[:nq], run.cache, run.block_tables[:n], run.context_lens[:n],
                      qsl, wl.num_heads, wl.scale, threads=threads)
        t_total += time.perf_counter() - t0
        reps += 1
    return {"value": round(reps * nbytes / t_total / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{n} of {wl.num_seqs} sequences (all heads), attention only, "
                      f"{reps} repetitions in {t_total:.1f} s"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step one bounded sample of the
    workload on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import workloads as W
    import oracle
    wl = W.NAMED[args.workload]()
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

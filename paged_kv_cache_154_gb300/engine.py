"""A paged KV cache for one attention layer, driven through the C ABI.

Holds the device cache tensors (torch allocations: the library itself
allocates nothing) and a host block pool, and runs the decode step in the
order the method requires: reserve slots in the pool (copy-on-write pairs
come back), copy the shared blocks, append the new K/V through the slot
mapping, then attend ("cs336 lecture 10", decode workflow: append the new
K, V, then score q against the cache).

Operations are duck-typed objects: one with `parent`/`child` is a fork, one
with `k`/`v` appends those rows to `seq`, anything else with `seq` creates a
sequence. Names are caller-chosen; `names` maps them to pool ids.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import (BLOCK_SIZE, Pool, append_kv, copy_blocks, decode, decode_shared_prefix,
               decode_shared_prefix_workspace_size, decode_workspace_size,
               zeroed_workspace)

KV_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "int8": torch.int8,
            "fp8": torch.float8_e4m3fn}


@dataclass
class StepInputs:
    """Device tensors of one decode step (built once, reusable)."""
    key: torch.Tensor                 # [T, H_kv, d] rows appended this step
    value: torch.Tensor
    slots: torch.Tensor               # int64 [T]
    pairs: Optional[torch.Tensor]     # int32 [n, 2] copy-on-write pairs, or None
    q: torch.Tensor                   # [num_q_tokens, H, d]
    block_tables: torch.Tensor        # int32 [S, max_blocks]
    context_lens: torch.Tensor        # int32 [S]
    query_start_loc: Optional[torch.Tensor]
    max_q_len: int
    max_context_len: int
    out: torch.Tensor
    workspace: Optional[torch.Tensor]
    shared: Optional["SharedPrefix"] = None


@dataclass
class SharedPrefix:
    """Fork groups of a step for read-once shared-prefix decode."""
    group_start: torch.Tensor         # int32 [G + 1] (device)
    prefix_len: torch.Tensor          # int32 [G] (device)
    group_start_host: np.ndarray
    prefix_len_host: np.ndarray
    max_group_q_len: int
    max_prefix_len: int
    workspace: torch.Tensor


class PagedKVCache:
    def __init__(self, num_blocks: int, num_kv_heads: int, head_dim: int, kv_dtype: str,
                 device="cuda", free_order: Optional[Sequence[int]] = None,
                 canary_blocks: int = 0, canary_byte: int = 0, head_scales=None):
        """head_scales: FP8 caches only, (k_scale, v_scale) per KV head (fp32,
        calibrated by the caller)."""
        self.num_blocks = num_blocks
        self.num_kv_heads = num_kv_heads
        self.head_dim = head_dim
        self.kv_dtype = kv_dtype
        self.device = torch.device(device)
        self.pool = Pool(num_blocks, BLOCK_SIZE, free_order)
        nb = num_blocks + canary_blocks
        shp = (nb, num_kv_heads, BLOCK_SIZE, head_dim)
        self.k = torch.zeros(shp, dtype=KV_TORCH[kv_dtype], device=self.device)
        self.v = torch.zeros(shp, dtype=KV_TORCH[kv_dtype], device=self.device)
        self.k_scale = self.v_scale = self.k_zp = self.v_zp = None
        if kv_dtype == "int8":
            self.k_scale = torch.zeros(shp[:3], dtype=torch.float32, device=self.device)
            self.v_scale = torch.zeros(shp[:3], dtype=torch.float32, device=self.device)
            self.k_zp = torch.zeros(shp[:3], dtype=torch.int8, device=self.device)
            self.v_zp = torch.zeros(shp[:3], dtype=torch.int8, device=self.device)
        if kv_dtype == "fp8":
            if head_scales is None:
                raise ValueError("an FP8 cache needs per-head scales (k_scale, v_scale)")
            ks, vs = head_scales
            self.k_scale = torch.as_tensor(np.asarray(ks, np.float32)).to(self.device)
            self.v_scale = torch.as_tensor(np.asarray(vs, np.float32)).to(self.device)
        if canary_blocks:
            for t in self.arrays():
                t[num_blocks:].view(torch.uint8).fill_(canary_byte)

    def arrays(self) -> List[torch.Tensor]:
        out = [self.k, self.v]
        if self.kv_dtype == "int8":
            out += [self.k_scale, self.v_scale, self.k_zp, self.v_zp]
        return out

    # -- host side of a phase: reserve slots, collect copy pairs --------------
    def reserve(self, ops, names: Dict) -> tuple:
        slots, pairs, ks, vs = [], [], [], []
        for op in ops:
            if hasattr(op, "parent"):
                names[op.child] = self.pool.seq_fork(names[op.parent])
            elif hasattr(op, "k"):
                sl, pair = self.pool.seq_append_slots(names[op.seq], int(op.k.shape[0]))
                if pair is not None:
                    pairs.append(pair)
                slots.append(sl)
                ks.append(op.k)
                vs.append(op.v)
            else:
                names[op.seq] = self.pool.seq_create()
        sl = np.concatenate(slots) if slots else np.zeros(0, np.int64)
        return sl, pairs, ks, vs

    # -- device side: copies first, then the append ------------------------------
    def write(self, slots: np.ndarray, pairs, ks, vs) -> None:
        if pairs:
            pr = torch.tensor(pairs, dtype=torch.int32, device=self.device)
            copy_blocks(self.k, self.v, pr, self.num_blocks, self.k_scale, self.v_scale,
                        self.k_zp, self.v_zp)
        if len(slots):
            key = torch.cat(ks).to(self.device)
            value = torch.cat(vs).to(self.device)
            sl = torch.from_numpy(np.ascontiguousarray(slots)).to(self.device)
            append_kv(key, value, self.k, self.v, sl, self.num_blocks, self.k_scale,
                      self.v_scale, self.k_zp, self.v_zp)

    def run_phase(self, ops, names: Dict) -> tuple:
        slots, pairs, ks, vs = self.reserve(ops, names)
        self.write(slots, pairs, ks, vs)
        return slots, pairs

    # -- decode step -------------------------------------------------------------
    def prepare_step(self, step_ops, names: Dict, q: torch.Tensor, out_dtype=torch.float32,
                     partition_size: int = 0, reserve: bool = True,
                     shared_prefix: bool = False) -> StepInputs:
        """Reserve the step's slots (host) and build its device inputs. With
        shared_prefix, also the fork groups (adjacent sequences of the step
        holding the same prompt blocks), so that attend_step reads each
        group's shared blocks once."""
        slots, pairs, ks, vs = self.reserve(step_ops, names) if reserve else (None, [], [], [])
        seqs = [names[op.seq] for op in step_ops]
        q_lens = [int(op.k.shape[0]) for op in step_ops]
        lens = [self.pool.seq_len(s) for s in seqs]
        max_blocks = max(1, max((L + BLOCK_SIZE - 1) // BLOCK_SIZE for L in lens))
        bt, cl = self.pool.block_tables(seqs, max_blocks)
        dev = self.device
        multi = max(q_lens) > 1
        qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
        nq = int(qsl[-1])
        ws_bytes = decode_workspace_size(len(seqs), nq, q.shape[1], self.num_kv_heads, q.shape[2],
                                         max(q_lens), max(lens), partition_size)
        shared = None
        if shared_prefix:
            gs, pl = self.pool.prefix_groups(seqs, q_lens)
            gq = [int(qsl[gs[g + 1]] - qsl[gs[g]]) for g in range(len(pl))]
            sp_bytes = decode_shared_prefix_workspace_size(
                len(seqs), nq, q.shape[1], self.num_kv_heads, q.shape[2], max(q_lens), max(lens),
                len(pl), max(gq), int(pl.max()), max_blocks)
            shared = SharedPrefix(
                group_start=torch.from_numpy(gs).to(dev), prefix_len=torch.from_numpy(pl).to(dev),
                group_start_host=gs, prefix_len_host=pl, max_group_q_len=max(gq),
                max_prefix_len=int(pl.max()),
                workspace=zeroed_workspace(sp_bytes, dev))
        return StepInputs(
            key=torch.cat(ks).to(dev), value=torch.cat(vs).to(dev),
            slots=torch.from_numpy(np.ascontiguousarray(slots)).to(dev),
            pairs=(torch.tensor(pairs, dtype=torch.int32, device=dev) if pairs else None),
            q=q.to(dev).contiguous(),
            block_tables=torch.from_numpy(bt).to(dev),
            context_lens=torch.from_numpy(cl).to(dev),
            query_start_loc=torch.from_numpy(qsl).to(dev) if multi else None,
            max_q_len=max(q_lens), max_context_len=max(lens),
            out=torch.empty((nq, q.shape[1], q.shape[2]), dtype=out_dtype, device=dev),
            workspace=zeroed_workspace(ws_bytes, dev),
            shared=shared)

    def write_step(self, si: StepInputs) -> None:
        """The step's cache writes: copy-on-write block copies, then the append."""
        if si.pairs is not None:
            copy_blocks(self.k, self.v, si.pairs, self.num_blocks, self.k_scale,
                        self.v_scale, self.k_zp, self.v_zp)
        append_kv(si.key, si.value, self.k, self.v, si.slots, self.num_blocks,
                  self.k_scale, self.v_scale, self.k_zp, self.v_zp)

    def attend_step(self, si: StepInputs, scale: float, partition_size: int = 0) -> torch.Tensor:
        """The step's attention over the cache (decode kernel + partial merge)."""
        if si.shared is not None:
            sp = si.shared
            decode_shared_prefix(si.out, si.q, self.k, self.v, si.block_tables, si.context_lens,
                                 si.max_context_len, scale, sp.group_start, sp.prefix_len,
                                 sp.max_group_q_len, sp.max_prefix_len, si.query_start_loc,
                                 si.max_q_len, self.num_blocks, sp.workspace)
            return si.out
        decode(si.out, si.q, self.k, self.v, si.block_tables, si.context_lens,
               si.max_context_len, scale, si.query_start_loc, si.max_q_len, self.num_blocks,
               self.k_scale, self.v_scale, self.k_zp, self.v_zp, partition_size,
               si.workspace)
        return si.out

    def step(self, si: StepInputs, scale: float, partition_size: int = 0,
             write: bool = True) -> torch.Tensor:
        """One decode step on device-resident inputs: copies, append, attend."""
        if write:
            self.write_step(si)
        return self.attend_step(si, scale, partition_size)

    def capture(self, fn, *args) -> "torch.cuda.CUDAGraph":
        """Record fn(*args) (e.g. write_step or attend_step) in a CUDA graph;
        graph.replay() then runs the same kernels on the same buffers with no
        per-launch host work. fn runs once eagerly first, so the library's
        one-time set-up (tensor maps, kernel attributes) happens outside the
        capture."""
        fn(*args)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(*args)
        torch.cuda.synchronize()
        return g

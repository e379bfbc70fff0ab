"""Seeded synthetic workloads for paged decode attention.

This module only makes inputs. It draws sequence lengths, speculative-verify
run lengths, the order of the free block list, the fork structure of
best-of-N groups, and N(0,1) values rounded (round-to-nearest-even) to the
storage dtype. It performs none of the method's arithmetic: no block-table
mapping, no slot computation, no attention and no quantisation. The CPU
oracle and the CUDA path both read the same objects it returns and never
import each other.

A workload is a *script* of host-side operations on a block pool (create a
sequence, fork it, append tokens with their K/V values) grouped in phases,
followed by one decode *step*: every decoding sequence appends its query-run
tokens and attends. Phases matter for copy-on-write: within one phase all
block copies are issued before any token is written, so a phase never
writes a block that another operation of the same phase copies from.

Shapes follow the pages' Llama-2/3-class models: 32 query / 8 KV heads with
head_dim 128 (Llama-3-8B, "ybb.press LLM推理优化深度实战" §2.2), 64 / 8
(Llama-2-70B GQA-8, "cs336 lecture 10" GQA section), MQA with one KV head
(same section), and 16-token blocks (page 1 "大模型推理优化全攻略" §2.3).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Union

import numpy as np
import torch

BLOCK_SIZE = 16
SEED_BASE = 1540

KV_DTYPES = ("f16", "bf16", "int8", "fp8")
TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Create:
    """Create an empty sequence named `seq` (a script-local name)."""
    seq: int


@dataclass
class Fork:
    """Make `child` share every block of `parent` (best-of-N sampling)."""
    parent: int
    child: int


@dataclass
class Append:
    """Append `k.shape[0]` tokens to `seq`; k, v are [n, H_kv, d] values."""
    seq: int
    k: torch.Tensor
    v: torch.Tensor

    @property
    def n(self) -> int:
        return int(self.k.shape[0])


Op = Union[Create, Fork, Append]


@dataclass
class Workload:
    name: str
    seed: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str                 # "f16" | "bf16" | "int8" (cache storage)
    src_dtype: torch.dtype        # dtype of the K/V values handed to append
    q_dtype: torch.dtype
    num_blocks: int
    free_order: np.ndarray        # int32 permutation: initial free list, popped from the end
    scale: float                  # softmax scale, an fp32 value
    phases: List[List[Op]]        # set-up phases (prefill, forks)
    step: List[Append]            # the decode step's appends, one per decoding sequence
    q: torch.Tensor               # [sum(q_lens), H_q, d], rows ordered like `step`
    context_lens: List[int]       # post-append lengths of the decoding sequences
    partition_size: int = 512
    block_size: int = BLOCK_SIZE
    notes: dict = field(default_factory=dict)
    head_scales: Optional[tuple] = None   # FP8 caches: (k_scale, v_scale), fp32 [H_kv] each

    @property
    def decode_seqs(self) -> List[int]:
        return [a.seq for a in self.step]

    @property
    def q_lens(self) -> List[int]:
        return [a.n for a in self.step]

    @property
    def num_seqs(self) -> int:
        return len(self.step)

    @property
    def max_context_len(self) -> int:
        return max(self.context_lens)

    @property
    def max_q_len(self) -> int:
        return max(self.q_lens)

    @property
    def query_start_loc(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    def total_tokens(self) -> int:
        n = 0
        for ph in self.phases:
            n += sum(op.n for op in ph if isinstance(op, Append))
        return n + sum(a.n for a in self.step)


class _Values:
    """N(0,1) fp32 draws from one seeded CPU generator, rounded RNE to a dtype."""

    def __init__(self, seed: int):
        self.g = torch.Generator(device="cpu")
        self.g.manual_seed(seed)

    def normal(self, shape, dtype: torch.dtype) -> torch.Tensor:
        return torch.randn(*shape, generator=self.g, dtype=torch.float32).to(dtype)


def _softmax_scale(head_dim: int) -> float:
    # the fp32 value of 1/sqrt(head_dim); both sides receive exactly this number
    return float(np.float32(1.0 / math.sqrt(head_dim)))


def _free_order(rng: np.random.Generator, num_blocks: int) -> np.ndarray:
    return rng.permutation(num_blocks).astype(np.int32)


def simple(name: str, seed: int, context_lens, q_lens, num_heads: int,
           num_kv_heads: int, head_dim: int, kv_dtype: str,
           q_dtype: torch.dtype = None, pool_factor: float = 1.2,
           min_pool_blocks: int = 0, key_row_boost: Optional[float] = None,
           boost_fraction: float = 0.01, partition_size: int = 512,
           value_scale: float = 1.0) -> Workload:
    """Independent sequences: prefill L - r tokens, then a step appending r.

    `context_lens` are post-append lengths (they include the step's r tokens).
    `key_row_boost`, when given, multiplies a seeded `boost_fraction` of the
    (token, kv_head) key rows by that factor (a power of two keeps the values
    exact in fp16/bf16), which makes the softmax peaked.
    """
    assert kv_dtype in KV_DTYPES
    context_lens = [int(x) for x in context_lens]
    q_lens = [int(x) for x in q_lens]
    assert len(context_lens) == len(q_lens)
    for L, r in zip(context_lens, q_lens):
        assert L >= r >= 1, (L, r)
    rng = np.random.default_rng(seed)
    vals = _Values(seed)
    src = torch.bfloat16 if kv_dtype in ("int8", "fp8") else TORCH_DTYPES[kv_dtype]
    if q_dtype is None:
        q_dtype = src
    need = sum((L + BLOCK_SIZE - 1) // BLOCK_SIZE for L in context_lens)
    num_blocks = max(int(math.ceil(pool_factor * need)), need, min_pool_blocks)
    free_order = _free_order(rng, num_blocks)

    def kv(n):
        k = vals.normal((n, num_kv_heads, head_dim), torch.float32)
        v = vals.normal((n, num_kv_heads, head_dim), torch.float32)
        if value_scale != 1.0:
            k = k * value_scale
            v = v * value_scale
        if key_row_boost is not None:
            rows = torch.from_numpy(rng.random((n, num_kv_heads)) < boost_fraction)
            k[rows] = k[rows] * key_row_boost
        return k.to(src), v.to(src)

    phase0: List[Op] = []
    step: List[Append] = []
    for s, (L, r) in enumerate(zip(context_lens, q_lens)):
        phase0.append(Create(s))
        if L - r > 0:
            k, v = kv(L - r)
            phase0.append(Append(s, k, v))
    for s, (L, r) in enumerate(zip(context_lens, q_lens)):
        k, v = kv(r)
        step.append(Append(s, k, v))
    q = vals.normal((sum(q_lens), num_heads, head_dim), q_dtype)
    return Workload(name=name, seed=seed, num_heads=num_heads,
                    num_kv_heads=num_kv_heads, head_dim=head_dim,
                    kv_dtype=kv_dtype, src_dtype=src, q_dtype=q_dtype,
                    num_blocks=num_blocks, free_order=free_order,
                    scale=_softmax_scale(head_dim), phases=[phase0], step=step,
                    q=q, context_lens=context_lens,
                    partition_size=partition_size,
                    head_scales=(calibrate_fp8([phase0], step, num_kv_heads)
                                 if kv_dtype == "fp8" else None))


FP8_MAX = 448.0   # largest finite E4M3 value


def calibrate_fp8(phases, step, num_kv_heads: int) -> tuple:
    """Per-KV-head FP8 scales from the data the workload will append (page 2
    "ybb.press" §5.2: per-head scaling factors found on calibration data):
    scale_h = max |x| over head h / 448, in fp32, separately for K and V, so
    no value saturates. Bookkeeping over generated values; no cache
    arithmetic."""
    amax = np.zeros((2, num_kv_heads), np.float64)
    for ops in list(phases) + [step]:
        for op in ops:
            if isinstance(op, Append):
                for i, t in enumerate((op.k, op.v)):
                    a = t.float().abs().amax(dim=(0, 2)).double().numpy()
                    amax[i] = np.maximum(amax[i], a)
    sc = np.where(amax > 0, amax / FP8_MAX, 1.0).astype(np.float32)
    return sc[0].copy(), sc[1].copy()


def best_of_n(name: str, seed: int, num_groups: int, n_forks: int,
              prompt_len: int, shared_extra_max: int, private_max: int,
              num_heads: int, num_kv_heads: int, head_dim: int,
              kv_dtype: str = "bf16", pool_factor: float = 1.2,
              partition_size: int = 512, step_q_max: int = 1) -> Workload:
    """Best-of-N groups sharing a prompt by refcount (copy-on-write).

    Each group has a parent holding `prompt_len + s` tokens, s in
    [1, shared_extra_max] (so its tail block is partial and shared), and
    `n_forks` children forked from it. The parent stays alive and is not
    decoded, so every child's first append into the shared tail copies it.
    Child 0 has no private tokens (its step append copies the tail); the
    others first append U[0, private_max] private tokens. The step appends one
    token to every child (or, with step_q_max > 1, a verify run of U[1,
    step_q_max] tokens) and decodes all children.
    """
    rng = np.random.default_rng(seed)
    vals = _Values(seed)
    src = torch.bfloat16 if kv_dtype in ("int8", "fp8") else TORCH_DTYPES[kv_dtype]
    s_extra = rng.integers(1, shared_extra_max + 1, size=num_groups)
    private = rng.integers(0, private_max + 1, size=(num_groups, n_forks))
    private[:, 0] = 0
    step_r = (np.ones((num_groups, n_forks), np.int64) if step_q_max == 1 else
              rng.integers(1, step_q_max + 1, size=(num_groups, n_forks)))
    need = 0
    for g in range(num_groups):
        plen = prompt_len + int(s_extra[g])
        need += (plen + BLOCK_SIZE - 1) // BLOCK_SIZE
        for i in range(n_forks):
            tail = int(s_extra[g]) + int(private[g, i]) + int(step_r[g, i])
            need += (tail + BLOCK_SIZE - 1) // BLOCK_SIZE
    num_blocks = int(math.ceil(pool_factor * need))
    free_order = _free_order(rng, num_blocks)

    def kv(n):
        k = vals.normal((n, num_kv_heads, head_dim), src)
        v = vals.normal((n, num_kv_heads, head_dim), src)
        return k, v

    phase0: List[Op] = []
    phase1: List[Op] = []
    step: List[Append] = []
    context_lens: List[int] = []
    nxt = 0
    children = []
    for g in range(num_groups):
        parent = nxt
        nxt += 1
        phase0.append(Create(parent))
        plen = prompt_len + int(s_extra[g])
        k, v = kv(plen)
        phase0.append(Append(parent, k, v))
        for i in range(n_forks):
            child = nxt
            nxt += 1
            phase1.append(Fork(parent, child))
            if private[g, i] > 0:
                k, v = kv(int(private[g, i]))
                phase1.append(Append(child, k, v))
            children.append((child, int(step_r[g, i])))
            context_lens.append(plen + int(private[g, i]) + int(step_r[g, i]))
    for child, r in children:
        k, v = kv(r)
        step.append(Append(child, k, v))
    q = vals.normal((int(step_r.sum()), num_heads, head_dim), src)
    return Workload(name=name, seed=seed, num_heads=num_heads,
                    num_kv_heads=num_kv_heads, head_dim=head_dim,
                    kv_dtype=kv_dtype, src_dtype=src, q_dtype=src,
                    num_blocks=num_blocks, free_order=free_order,
                    scale=_softmax_scale(head_dim), phases=[phase0, phase1],
                    step=step, q=q, context_lens=context_lens,
                    partition_size=partition_size,
                    notes={"shared_extra": s_extra.tolist(),
                           "private": private.tolist()},
                    head_scales=(calibrate_fp8([phase0, phase1], step, num_kv_heads)
                                 if kv_dtype == "fp8" else None))


# --------------------------------------------------------------------------
# The five named workloads (sizes as stated in their docstrings).
# --------------------------------------------------------------------------

# Shard r of a workload (one per rank when several GPUs each take their own
# batch of independent sequences) draws from seed + SHARD_STRIDE * r; shard 0
# is the workload itself.
SHARD_STRIDE = 1000


def tiny(shard: int = 0) -> Workload:
    """4 sequences, post-append lengths {17, 33, 64, 100}; 8 q / 2 KV heads,
    head_dim 64, fp16, a 64-block pool placed by a seeded permutation."""
    return simple("tiny", SEED_BASE + 1 + SHARD_STRIDE * shard, [17, 33, 64, 100],
                  [1, 1, 1, 1], num_heads=8, num_kv_heads=2, head_dim=64, kv_dtype="f16",
                  pool_factor=0.0, min_pool_blocks=64)


def llama3_8b(batch: int = 64, lo: int = 512, hi: int = 4096, shard: int = 0) -> Workload:
    """Llama-3-8B-shaped decode step: 64 sequences, lengths U[512, 4096],
    32 q / 8 KV heads, head_dim 128, bf16, pool 1.2x the blocks needed."""
    seed = SEED_BASE + 2 + SHARD_STRIDE * shard
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=batch)
    return simple("llama3_8b_decode", seed, lens, [1] * batch,
                  num_heads=32, num_kv_heads=8, head_dim=128, kv_dtype="bf16")


def llama3_8b_fp8(batch: int = 64, lo: int = 512, hi: int = 4096, shard: int = 0) -> Workload:
    """The Llama-3-8B-shaped decode step with an FP8 (E4M3) cache: 64
    sequences, lengths U[512, 4096], 32 q / 8 KV heads, head_dim 128, bf16 q,
    per-head scales calibrated on the appended data."""
    seed = SEED_BASE + 6 + SHARD_STRIDE * shard
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=batch)
    return simple("llama3_8b_fp8", seed, lens, [1] * batch, num_heads=32, num_kv_heads=8,
                  head_dim=128, kv_dtype="fp8", q_dtype=torch.bfloat16)


def paged_prefill(batch: int = 8, chunk: int = 512, prior_max: int = 4096,
                  shard: int = 0) -> Workload:
    """Chunked prefill over the paged cache, Llama-3-8B-shaped (32 q / 8 KV
    heads, head_dim 128, bf16): 8 sequences that already hold U[0, 4096]
    cached tokens each append a chunk of 512 prompt tokens and attend them
    causally (query i of the chunk sees the prior tokens and chunk tokens
    0 .. i): 2048 query rows per KV head."""
    seed = SEED_BASE + 7 + SHARD_STRIDE * shard
    rng = np.random.default_rng(seed)
    prior = rng.integers(0, prior_max + 1, size=batch)
    return simple("paged_prefill_llama3_8b", seed, prior + chunk, [chunk] * batch,
                  num_heads=32, num_kv_heads=8, head_dim=128, kv_dtype="bf16")


def llama2_70b_best_of_5(num_groups: int = 8, prompt_len: int = 4096,
                         shard: int = 0) -> Workload:
    """Llama-2-70B-shaped best-of-5: 8 prompts of 4096 (+1..15 shared) tokens,
    forked 5 ways, 0-256 private tokens per fork, 64 q / 8 KV heads, bf16."""
    return best_of_n("llama2_70b_best_of_5", SEED_BASE + 3 + SHARD_STRIDE * shard,
                     num_groups, 5, prompt_len, 15, 256, num_heads=64, num_kv_heads=8,
                     head_dim=128)


def long_context(lens=(32768, 65536, 100000, 131072), shard: int = 0) -> Workload:
    """Long-context split-KV decode: 4 sequences up to 131072 tokens, 32 q /
    8 KV heads, head_dim 128, bf16, 1% of key rows scaled by 8."""
    return simple("long_context_split_kv", SEED_BASE + 4 + SHARD_STRIDE * shard, list(lens),
                  [1] * len(lens), num_heads=32, num_kv_heads=8, head_dim=128,
                  kv_dtype="bf16", pool_factor=1.05, key_row_boost=8.0)


def mixed_int8(batch: int = 256, median: int = 1024, cap: int = 16384,
               verify_fraction: float = 0.2, shard: int = 0,
               name: str = "mixed_mqa_int8_verify") -> Workload:
    """Continuous-batching mixed step: 256 sequences with lognormal lengths
    (median 1024, sigma 1, capped at 16384), MQA 32 q / 1 KV head, head_dim
    128, INT8 KV; 20% of sequences carry a verify run of 2-5 query tokens."""
    seed = SEED_BASE + 5 + SHARD_STRIDE * shard
    rng = np.random.default_rng(seed)
    raw = rng.lognormal(mean=math.log(median), sigma=1.0, size=batch)
    q_lens = np.ones(batch, dtype=np.int64)
    nver = int(round(verify_fraction * batch))
    ver = rng.choice(batch, size=nver, replace=False)
    q_lens[ver] = rng.integers(2, 6, size=nver)
    lens = np.minimum(np.rint(raw), cap).astype(np.int64)
    lens = np.maximum(lens, q_lens)
    return simple(name, seed, lens, q_lens,
                  num_heads=32, num_kv_heads=1, head_dim=128, kv_dtype="int8",
                  q_dtype=torch.bfloat16)


def mqa_int8_verify(shard: int = 0) -> Workload:
    """Speculative-decoding verify step over an INT8 cache: the mixed step's
    256 sequences and lengths with every sequence verifying 2-5 draft tokens
    (64-160 query rows per KV head; MQA 32 q / 1 KV head, head_dim 128)."""
    return mixed_int8(verify_fraction=1.0, shard=shard, name="mqa_int8_verify_all")


NAMED = {
    "tiny": tiny,
    "llama3_8b": llama3_8b,
    "llama2_70b_best_of_5": llama2_70b_best_of_5,
    "long_context": long_context,
    "mixed_int8": mixed_int8,
    "mqa_int8_verify": mqa_int8_verify,
    "llama3_8b_fp8": llama3_8b_fp8,
    "paged_prefill": paged_prefill,
}


# --------------------------------------------------------------------------
# Bookkeeping over generated values (no arithmetic on them)
# --------------------------------------------------------------------------

CANARY_BLOCKS = 2      # guard blocks after the pool; filled with CANARY_BYTE, never written
CANARY_BYTE = 0x7E


def contiguous_kv(wl: Workload):
    """Per decoding sequence, the K and V it holds in token order, [L, H_kv, d]:
    the concatenation of every Append made to it (a fork inherits its parent's
    tokens at fork time). This is the data before any paging."""
    chunks = {}
    for ph in wl.phases + [wl.step]:
        for op in ph:
            if isinstance(op, Create):
                chunks[op.seq] = []
            elif isinstance(op, Fork):
                chunks[op.child] = list(chunks[op.parent])
            elif isinstance(op, Append):
                chunks[op.seq].append((op.k, op.v))
    out = []
    for a in wl.step:
        ks = [k for k, _ in chunks[a.seq]]
        vs = [v for _, v in chunks[a.seq]]
        out.append((torch.cat(ks, 0), torch.cat(vs, 0)))
    return out


def with_free_order(wl: Workload, seed: int) -> Workload:
    """The same workload with another seeded placement of physical blocks."""
    import dataclasses
    rng = np.random.default_rng(seed)
    return dataclasses.replace(wl, free_order=_free_order(rng, wl.num_blocks))

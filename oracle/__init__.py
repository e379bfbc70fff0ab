"""CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import this package. It never imports the CUDA library or its binding, and
the CUDA library never imports it; the two share only the seeded input
generators in `workloads`.

Contents (each function cites the passage it restates):
  * oracle.c      -- fp64 attention over a paged cache, append scatter, INT8
                     quantiser (fp32), block copies; built with gcc.
  * allocator.py  -- block pool with refcounts and copy-on-write.
  * formulas.py   -- the KV-cache memory formula.
  * lse_merge()   -- the split-KV log-sum-exp merge (below).
  * run()         -- executes a workload script sequentially on the host.

Parity pins for every function live in tests/test_oracle_*.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np

from .allocator import BlockPool, OutOfBlocks  # noqa: F401
from . import formulas  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DTYPE_CODE = {"f16": 0, "bf16": 1, "f32": 2, "int8": 3, "fp8": 4}


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/liboracle.so (gcc, OpenMP, IEEE fp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        L.orc_attend.argtypes = [P, P, P, P, P, P, ctypes.c_int, P, P, P, P, P,
                                 ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, f64,
                                 i64, i64, ctypes.c_int]
        L.orc_attend.restype = ctypes.c_int
        L.orc_append.argtypes = [P, P, P, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.orc_append.restype = None
        L.orc_append_int8.argtypes = [P, P, P, P, ctypes.c_int, P, i64, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int]
        L.orc_append_int8.restype = None
        L.orc_quantize_row.argtypes = [P, ctypes.c_int, P, P, P]
        L.orc_quantize_row.restype = None
        L.orc_copy_blocks.argtypes = [P, i64, P, ctypes.c_int]
        L.orc_copy_blocks.restype = None
        L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_f64.restype = f64
        L.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_to_f64.restype = f64
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_append_fp8.argtypes = [P, P, P, ctypes.c_int, P, i64, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int]
        L.orc_append_fp8.restype = None
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------
# host cache
# ---------------------------------------------------------------------------

@dataclass
class HostCache:
    """Host copy of one layer's paged cache, [num_blocks][H_kv][block_size][d]."""
    kv_dtype: str
    k: np.ndarray
    v: np.ndarray
    k_scale: Optional[np.ndarray] = None
    v_scale: Optional[np.ndarray] = None
    k_zp: Optional[np.ndarray] = None
    v_zp: Optional[np.ndarray] = None

    @property
    def num_blocks(self) -> int:
        return self.k.shape[0]

    @property
    def num_kv_heads(self) -> int:
        return self.k.shape[1]

    @property
    def block_size(self) -> int:
        return self.k.shape[2]

    @property
    def head_dim(self) -> int:
        return self.k.shape[3]

    def arrays(self):
        """The per-block arrays (what a block copy copies and the cache
        comparison compares); FP8's per-head scales are not per block."""
        out = [self.k, self.v]
        if self.kv_dtype == "int8":
            out += [self.k_scale, self.v_scale, self.k_zp, self.v_zp]
        return out


def empty_cache(kv_dtype: str, num_blocks: int, num_kv_heads: int,
                block_size: int, head_dim: int, canary_blocks: int = 0,
                canary_byte: int = 0, head_scales=None) -> HostCache:
    """Zeroed cache of num_blocks + canary_blocks blocks; the trailing canary
    blocks are filled with canary_byte (they must never change). FP8 caches
    take head_scales = (k_scale, v_scale), fp32 [num_kv_heads] each."""
    nb = num_blocks + canary_blocks
    shp = (nb, num_kv_heads, block_size, head_dim)
    if kv_dtype == "int8":
        c = HostCache("int8", np.zeros(shp, np.int8), np.zeros(shp, np.int8),
                      np.zeros(shp[:3], np.float32), np.zeros(shp[:3], np.float32),
                      np.zeros(shp[:3], np.int8), np.zeros(shp[:3], np.int8))
    elif kv_dtype == "fp8":
        ks, vs = head_scales
        c = HostCache("fp8", np.zeros(shp, np.uint8), np.zeros(shp, np.uint8),
                      np.ascontiguousarray(ks, dtype=np.float32),
                      np.ascontiguousarray(vs, dtype=np.float32))
    else:
        c = HostCache(kv_dtype, np.zeros(shp, np.uint16), np.zeros(shp, np.uint16))
    if canary_blocks:
        for a in c.arrays():
            a[num_blocks:].view(np.uint8)[...] = canary_byte
    return c


def _bits16(t) -> np.ndarray:
    """Raw 16-bit patterns of a torch fp16/bf16 tensor (no conversion)."""
    import torch
    return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def append(cache: HostCache, k_src, v_src, slots: np.ndarray, src_dtype: str) -> None:
    """Scatter new rows [T, H_kv, d] into the cache at `slots` (negative = skip).
    Page 4 ("cs336 lecture 10"), KV Cache workflow: append the new K and V."""
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    T = slots.shape[0]
    kb, vb = _bits16(k_src), _bits16(v_src)
    assert kb.shape == (T, cache.num_kv_heads, cache.head_dim)
    L = lib()
    if cache.kv_dtype == "fp8":
        for src, codes, sc in ((kb, cache.k, cache.k_scale), (vb, cache.v, cache.v_scale)):
            L.orc_append_fp8(_p(codes), _p(sc), _p(src), DTYPE_CODE[src_dtype], _p(slots), T,
                             cache.num_kv_heads, cache.head_dim, cache.block_size)
    elif cache.kv_dtype == "int8":
        for src, codes, sc, zp in ((kb, cache.k, cache.k_scale, cache.k_zp),
                                   (vb, cache.v, cache.v_scale, cache.v_zp)):
            L.orc_append_int8(_p(codes), _p(sc), _p(zp), _p(src), DTYPE_CODE[src_dtype],
                              _p(slots), T, cache.num_kv_heads, cache.head_dim,
                              cache.block_size)
    else:
        for src, dst in ((kb, cache.k), (vb, cache.v)):
            L.orc_append(_p(dst), _p(src), _p(slots), T, cache.num_kv_heads,
                         cache.head_dim, cache.block_size)


def copy_blocks(cache: HostCache, pairs: List[Tuple[int, int]]) -> None:
    """Copy whole physical blocks src -> dst in every cache array
    (page 2 "ybb.press" §2.1: copy only when a shared block is modified)."""
    if not pairs:
        return
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    for a in cache.arrays():
        per_block = a[0].nbytes
        lib().orc_copy_blocks(_p(a), per_block, _p(pr), pr.shape[0])


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """FP8 E4M3 code -> value (fp64), from the format's definition."""
    L = lib()
    flat = np.asarray(codes, dtype=np.uint8).reshape(-1)
    return np.array([L.orc_e4m3_to_f64(int(c)) for c in flat]).reshape(np.shape(codes))


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """fp32 values -> nearest FP8 E4M3 codes (ties to even, saturating at 448)."""
    L = lib()
    flat = np.asarray(x, dtype=np.float32).reshape(-1)
    return np.array([L.orc_e4m3_encode(float(v)) for v in flat],
                    dtype=np.uint8).reshape(np.shape(x))


def quantize_row(x: np.ndarray) -> Tuple[np.ndarray, float, int]:
    """INT8 quantiser of one row (page 4 "cs336 lecture 10", Quantization:
    x_q = round(x / scale) + zero_point), fp32 arithmetic."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.zeros(x.shape[0], np.int8)
    sc = np.zeros(1, np.float32)
    zp = np.zeros(1, np.int8)
    lib().orc_quantize_row(_p(x), x.shape[0], _p(codes), _p(sc), _p(zp))
    return codes, float(sc[0]), int(zp[0])


def dequantize(codes: np.ndarray, scale, zp) -> np.ndarray:
    """x = (x_q - zero_point) * scale, one fp32 rounding (same page)."""
    c = codes.astype(np.int32) - np.asarray(zp, dtype=np.int32)
    return (c.astype(np.float32) * np.asarray(scale, dtype=np.float32)).astype(np.float32)


def attend(q64: np.ndarray, cache: HostCache, block_tables: np.ndarray,
           context_lens: np.ndarray, query_start_loc: Optional[np.ndarray],
           num_heads: int, scale: float, t_begin: int = 0,
           t_end: Optional[int] = None, threads: int = 1):
    """fp64 softmax(scale * q K^T) V over the keys each query sees within
    [t_begin, t_end). Returns (o, m, l): o normalised, m the max logit and l
    the sum of exp(logit - m) (page 3 §二 attention formula; page 4 decode
    workflow; GQA: q head h reads kv head h // (H_q / H_kv))."""
    q64 = np.ascontiguousarray(q64, dtype=np.float64)
    T = q64.shape[0]
    o = np.zeros((T, num_heads, cache.head_dim), np.float64)
    m = np.zeros((T, num_heads), np.float64)
    l = np.zeros((T, num_heads), np.float64)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qsl = None if query_start_loc is None else np.ascontiguousarray(query_start_loc, dtype=np.int32)
    if t_end is None:
        t_end = 1 << 62
    rc = lib().orc_attend(_p(o), _p(m), _p(l), _p(q64), _p(cache.k), _p(cache.v),
                          DTYPE_CODE[cache.kv_dtype], _p(cache.k_scale), _p(cache.v_scale),
                          _p(cache.k_zp), _p(cache.v_zp), _p(bt), bt.shape[1], _p(cl),
                          _p(qsl), cl.shape[0], num_heads, cache.num_kv_heads,
                          cache.head_dim, cache.block_size, float(scale), int(t_begin),
                          int(t_end), int(threads))
    if rc != 0:
        raise ValueError(f"oracle attend rejected its input (code {rc})")
    return o, m, l


def lse_merge(o_parts: np.ndarray, m_parts: np.ndarray, l_parts: np.ndarray) -> np.ndarray:
    """Merge split-KV partitions: out = sum_p w_p o_p / sum_p w_p with
    w_p = l_p exp(m_p - M), M = max_p m_p (the log-sum-exp rescaling that
    makes a softmax over a union of key sets from per-set results).
    Shapes: o_parts [P, ..., d], m_parts / l_parts [P, ...]."""
    M = np.max(m_parts, axis=0)
    Msafe = np.where(np.isfinite(M), M, 0.0)
    with np.errstate(invalid="ignore"):
        w = np.where(l_parts > 0, l_parts * np.exp(m_parts - Msafe), 0.0)
    den = np.sum(w, axis=0)
    num = np.sum(w[..., None] * o_parts, axis=0)
    return num / den[..., None]


# ---------------------------------------------------------------------------
# running a workload script on the host
# ---------------------------------------------------------------------------

@dataclass
class Run:
    pool: BlockPool
    cache: HostCache
    names: dict                    # script name -> pool sequence id
    phase_slots: List[np.ndarray]  # slots of each phase, concatenated in op order
    phase_pairs: List[list]        # copy pairs of each phase, in op order
    step_slots: np.ndarray
    step_pairs: list
    block_tables: np.ndarray       # [S, max_blocks] int32, padded with -1
    context_lens: np.ndarray
    q64: np.ndarray
    out: Optional[np.ndarray] = None
    extra: dict = field(default_factory=dict)


def _run_ops(pool, cache, names, ops, src_dtype):
    from workloads import Append, Create, Fork
    slots_all, pairs = [], []
    for op in ops:
        if isinstance(op, Create):
            names[op.seq] = pool.create()
        elif isinstance(op, Fork):
            names[op.child] = pool.fork(names[op.parent])
        elif isinstance(op, Append):
            slots, pair = pool.append_slots(names[op.seq], op.n)
            if pair is not None:
                copy_blocks(cache, [pair])
                pairs.append(pair)
            sl = np.asarray(slots, np.int64)
            append(cache, op.k, op.v, sl, src_dtype)
            slots_all.append(sl)
        else:
            raise TypeError(op)
    sl = np.concatenate(slots_all) if slots_all else np.zeros(0, np.int64)
    return sl, pairs


def run(wl, threads: int = 1, canary_blocks: int = 0, canary_byte: int = 0,
        decode: bool = True) -> Run:
    """Execute the workload's phases and step one operation at a time (block
    copies before that operation's write), then attend."""
    src_dtype = {"torch.float16": "f16", "torch.bfloat16": "bf16"}[str(wl.src_dtype)]
    pool = BlockPool(wl.num_blocks, wl.block_size, wl.free_order)
    cache = empty_cache(wl.kv_dtype, wl.num_blocks, wl.num_kv_heads, wl.block_size,
                        wl.head_dim, canary_blocks, canary_byte,
                        head_scales=getattr(wl, "head_scales", None))
    names: dict = {}
    ph_slots, ph_pairs = [], []
    for ops in wl.phases:
        s, p = _run_ops(pool, cache, names, ops, src_dtype)
        ph_slots.append(s)
        ph_pairs.append(p)
    st_slots, st_pairs = _run_ops(pool, cache, names, wl.step, src_dtype)
    seqs = [names[a.seq] for a in wl.step]
    max_blocks = max(len(pool.block_table(s)) for s in seqs)
    bt = np.full((len(seqs), max_blocks), -1, np.int32)
    for i, s in enumerate(seqs):
        t = pool.block_table(s)
        bt[i, :len(t)] = t
    cl = np.asarray([pool.lens[s] for s in seqs], np.int32)
    q64 = wl.q.double().numpy()
    r = Run(pool, cache, names, ph_slots, ph_pairs, st_slots, st_pairs, bt, cl, q64)
    if decode:
        r.out, r.extra["m"], r.extra["l"] = attend(
            q64, cache, bt, cl, wl.query_start_loc, wl.num_heads, wl.scale,
            threads=threads)
    return r

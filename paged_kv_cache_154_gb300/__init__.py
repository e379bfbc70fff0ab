"""Python binding of libpa.so, the paged KV-cache decode-attention library.

Argument marshalling only: every function here forwards torch tensors as raw
device pointers to the C ABI declared in include/pa.h (same names, without
the `pa_` prefix), on the current CUDA stream, and raises PAError on a
non-zero status. Every step of the computation runs in the library's CUDA
kernels; there is no Python or CPU fallback. If libpa.so has not been built
(`python -m paged_kv_cache_154_gb300.build`), importing the functions fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")

PA_F16, PA_BF16, PA_F32, PA_INT8, PA_FP8_E4M3 = 0, 1, 2, 3, 4
STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED",
          3: "PA_ERR_OUT_OF_BLOCKS", 4: "PA_ERR_BAD_REFCOUNT", 5: "PA_ERR_CUDA",
          6: "PA_ERR_VALIDATION", 7: "PA_ERR_DEVICE"}
BLOCK_SIZE = 16


class PAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None
_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t

_SIGS = {
    "pa_last_error": ([], ctypes.c_char_p),
    "pa_version": ([], ctypes.c_char_p),
    "pa_pool_create": ([_I32, _I32, _P, ctypes.POINTER(_P)], ctypes.c_int),
    "pa_pool_destroy": ([_P], None),
    "pa_seq_create": ([_P, _P], ctypes.c_int),
    "pa_seq_fork": ([_P, _I32, _P], ctypes.c_int),
    "pa_seq_append_slots": ([_P, _I32, _I32, _P, _P, _P], ctypes.c_int),
    "pa_seq_append_slots_batch": ([_P, _P, _P, _I32, _P, _P, _P], ctypes.c_int),
    "pa_seq_free": ([_P, _I32], ctypes.c_int),
    "pa_seq_len": ([_P, _I32, _P], ctypes.c_int),
    "pa_pool_block_tables": ([_P, _P, _I32, _I32, _P, _P], ctypes.c_int),
    "pa_pool_stats": ([_P, _P, _P, _P], ctypes.c_int),
    "pa_pool_refcount": ([_P, _I32, _P], ctypes.c_int),
    "pa_copy_blocks": ([_P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32,
                        ctypes.c_int, _P], ctypes.c_int),
    "pa_append_kv": ([_P, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P, _P, _P, _P,
                      _I32, _I32, _I32, _I32, _I32, _P], ctypes.c_int),
    "pa_decode_workspace_size": ([_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32], _SZ),
    "pa_decode": ([_P, ctypes.c_int, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P, _P, _P,
                   _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                   ctypes.c_float, _I32, _I32, _P, _SZ, _P], ctypes.c_int),
    "pa_decode_no_alloc": ([_P, ctypes.c_int, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P,
                            _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                            _I32, ctypes.c_float, _I32, _I32, _P], ctypes.c_int),
    "pa_device_error": ([_P, _P], ctypes.c_int),
    "pa_pool_prefix_groups": ([_P, _P, _I32, _P, _P, _P, _P], ctypes.c_int),
    "pa_pool_enable_prefix_cache": ([_P, _I32], ctypes.c_int),
    "pa_seq_create_with_prefix": ([_P, _P, _I32, _P, _P], ctypes.c_int),
    "pa_seq_append_tokens": ([_P, _I32, _P, _I32, _P, _P, _P], ctypes.c_int),
    "pa_pool_prefix_stats": ([_P, _P, _P, _P, _P], ctypes.c_int),
    "pa_decode_shared_prefix_workspace_size": ([_I32] * 11, _SZ),
    "pa_decode_shared_prefix": ([_P, ctypes.c_int, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P,
                                 _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                                 ctypes.c_float, _I32, _P, _P, _I32, _I32, _I32, _P, _SZ, _P],
                                ctypes.c_int),
}


def lib() -> ctypes.CDLL:
    """The loaded libpa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_cache_154_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise PAError(status, lib().pa_last_error().decode())


def version() -> str:
    return lib().pa_version().decode()


def _dtype_code(t) -> int:
    import torch
    return {torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.float32: PA_F32,
            torch.int8: PA_INT8, torch.float8_e4m3fn: PA_FP8_E4M3}[t.dtype]


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    assert t.is_contiguous(), "tensors passed to libpa must be contiguous"
    return t.data_ptr()


def _stream(stream=None) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


# ---------------------------------------------------------------------------
# host block pool
# ---------------------------------------------------------------------------

class Pool:
    """pa_pool_*: block pool with refcounts and copy-on-write (host memory)."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE,
                 free_order: Optional[Sequence[int]] = None):
        self._h = _P()
        fo = None
        if free_order is not None:
            self._fo = np.ascontiguousarray(free_order, dtype=np.int32)
            fo = self._fo.ctypes.data
        _check(lib().pa_pool_create(num_blocks, block_size, fo, ctypes.byref(self._h)))
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.pa_pool_destroy(self._h)
            self._h = None

    def seq_create(self) -> int:
        out = _I32()
        _check(lib().pa_seq_create(self._h, ctypes.addressof(out)))
        return out.value

    def seq_fork(self, parent: int) -> int:
        out = _I32()
        _check(lib().pa_seq_fork(self._h, parent, ctypes.addressof(out)))
        return out.value

    def seq_append_slots(self, seq: int, n: int) -> Tuple[np.ndarray, Optional[Tuple[int, int]]]:
        slots = np.zeros(max(n, 1), np.int64)
        pair = np.zeros(2, np.int32)
        ncow = _I32()
        _check(lib().pa_seq_append_slots(self._h, seq, n, slots.ctypes.data, pair.ctypes.data,
                                         ctypes.addressof(ncow)))
        return slots[:n], ((int(pair[0]), int(pair[1])) if ncow.value else None)

    def seq_append_slots_batch(self, seqs: Sequence[int], counts: Sequence[int],
                               slots_out: Optional[np.ndarray] = None
                               ) -> Tuple[np.ndarray, np.ndarray]:
        """One step's reservations in one call (pa_seq_append_slots_batch):
        the slots of every sequence in order (into slots_out if given, int64
        [sum(counts)]) and the copy-on-write pairs, int32 [k][2]."""
        s = np.ascontiguousarray(seqs, dtype=np.int32)
        c = np.ascontiguousarray(counts, dtype=np.int32)
        total = int(c.sum())
        slots = slots_out if slots_out is not None else np.zeros(max(total, 1), np.int64)
        pairs = np.zeros((max(len(s), 1), 2), np.int32)
        ncow = _I32()
        _check(lib().pa_seq_append_slots_batch(self._h, s.ctypes.data, c.ctypes.data, len(s),
                                               slots.ctypes.data, pairs.ctypes.data,
                                               ctypes.addressof(ncow)))
        return slots[:total], pairs[:ncow.value]

    def seq_free(self, seq: int) -> None:
        _check(lib().pa_seq_free(self._h, seq))

    def seq_len(self, seq: int) -> int:
        out = _I32()
        _check(lib().pa_seq_len(self._h, seq, ctypes.addressof(out)))
        return out.value

    def block_tables(self, seqs: Sequence[int], max_blocks: int) -> Tuple[np.ndarray, np.ndarray]:
        s = np.ascontiguousarray(seqs, dtype=np.int32)
        tables = np.zeros((len(s), max_blocks), np.int32)
        lens = np.zeros(len(s), np.int32)
        _check(lib().pa_pool_block_tables(self._h, s.ctypes.data, len(s), max_blocks,
                                          tables.ctypes.data, lens.ctypes.data))
        return tables, lens

    def stats(self) -> Tuple[int, int, int]:
        f, u, sh = _I32(), _I32(), _I32()
        _check(lib().pa_pool_stats(self._h, ctypes.addressof(f), ctypes.addressof(u),
                                   ctypes.addressof(sh)))
        return f.value, u.value, sh.value

    def refcount(self, block: int) -> int:
        out = _I32()
        _check(lib().pa_pool_refcount(self._h, block, ctypes.addressof(out)))
        return out.value

    # -- prefix cache ------------------------------------------------------
    def enable_prefix_cache(self, max_cached_blocks: int) -> None:
        _check(lib().pa_pool_enable_prefix_cache(self._h, int(max_cached_blocks)))

    def create_with_prefix(self, token_ids: Sequence[int]) -> Tuple[int, int]:
        """pa_seq_create_with_prefix: (sequence id, tokens already cached)."""
        t = np.ascontiguousarray(token_ids, dtype=np.int32)
        sid, n = _I32(), _I32()
        _check(lib().pa_seq_create_with_prefix(self._h, t.ctypes.data if len(t) else None,
                                               len(t), ctypes.addressof(sid),
                                               ctypes.addressof(n)))
        return sid.value, n.value

    def append_tokens(self, seq: int, token_ids: Sequence[int]
                      ) -> Tuple[np.ndarray, Optional[Tuple[int, int]]]:
        """pa_seq_append_tokens: (slots, copy pair or None)."""
        t = np.ascontiguousarray(token_ids, dtype=np.int32)
        slots = np.zeros(max(1, len(t)), np.int64)
        pair = np.zeros(2, np.int32)
        ncow = _I32()
        _check(lib().pa_seq_append_tokens(self._h, seq, t.ctypes.data if len(t) else None,
                                          len(t), slots.ctypes.data, pair.ctypes.data,
                                          ctypes.addressof(ncow)))
        return slots[:len(t)].copy(), ((int(pair[0]), int(pair[1])) if ncow.value else None)

    def prefix_stats(self) -> Tuple[int, int, int, int]:
        """(cached unreferenced blocks, registered blocks, hit blocks, looked-up blocks)."""
        c, r = _I32(), _I32()
        h, l = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().pa_pool_prefix_stats(self._h, ctypes.addressof(c), ctypes.addressof(r),
                                          ctypes.addressof(h), ctypes.addressof(l)))
        return c.value, r.value, h.value, l.value

    def prefix_groups(self, seqs: Sequence[int],
                      q_lens: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
        """pa_pool_prefix_groups: (group_start [G + 1], prefix_len [G]) for the
        sequences in this order (adjacent forks of one prompt form a group)."""
        s = np.ascontiguousarray(seqs, dtype=np.int32)
        ql = None if q_lens is None else np.ascontiguousarray(q_lens, dtype=np.int32)
        gs = np.zeros(len(s) + 1, np.int32)
        pl = np.zeros(max(1, len(s)), np.int32)
        ng = _I32()
        _check(lib().pa_pool_prefix_groups(self._h, s.ctypes.data, len(s),
                                           None if ql is None else ql.ctypes.data,
                                           gs.ctypes.data, pl.ctypes.data,
                                           ctypes.addressof(ng)))
        return gs[:ng.value + 1].copy(), pl[:ng.value].copy()


# ---------------------------------------------------------------------------
# device operations (torch tensors in, nothing allocated)
# ---------------------------------------------------------------------------

def copy_blocks(k_cache, v_cache, pairs, num_blocks: Optional[int] = None, k_scale=None,
                v_scale=None, k_zp=None, v_zp=None, stream=None) -> None:
    """pa_copy_blocks; pairs: device int32 [n, 2] (src, dst)."""
    n = 0 if pairs is None else int(pairs.shape[0])
    if n == 0:
        return
    nb = k_cache.shape[0] if num_blocks is None else num_blocks
    _check(lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                _ptr(k_zp), _ptr(v_zp), _ptr(pairs), n, nb,
                                k_cache.shape[1], k_cache.shape[3], k_cache.shape[2],
                                _dtype_code(k_cache), _stream(stream)))


def append_kv(key, value, k_cache, v_cache, slot_mapping, num_blocks: Optional[int] = None,
              k_scale=None, v_scale=None, k_zp=None, v_zp=None, stream=None) -> None:
    """pa_append_kv; key/value [T, H_kv, d]; slot_mapping device int64 [T]."""
    T = int(key.shape[0])
    nb = k_cache.shape[0] if num_blocks is None else num_blocks
    _check(lib().pa_append_kv(_ptr(key), _ptr(value), _dtype_code(key), _ptr(k_cache),
                              _ptr(v_cache), _dtype_code(k_cache), _ptr(k_scale),
                              _ptr(v_scale), _ptr(k_zp), _ptr(v_zp), _ptr(slot_mapping), T, nb,
                              k_cache.shape[1], k_cache.shape[3], k_cache.shape[2],
                              _stream(stream)))


def decode_workspace_size(num_seqs: int, num_q_tokens: int, num_heads: int, num_kv_heads: int,
                          head_dim: int, max_q_len: int, max_context_len: int,
                          partition_size: int = 0) -> int:
    return int(lib().pa_decode_workspace_size(num_seqs, num_q_tokens, num_heads, num_kv_heads,
                                              head_dim, max_q_len, max_context_len,
                                              partition_size))


def zeroed_workspace(nbytes: int, device="cuda"):
    """A decode workspace of `nbytes` (from decode_workspace_size or
    decode_shared_prefix_workspace_size): zero-filled as the arrival counters
    at its start require, 256-byte aligned (torch's allocator), None for 0."""
    import torch
    if nbytes <= 0:
        return None
    return torch.zeros(int(nbytes), dtype=torch.uint8, device=device)


def decode(out, q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
           scale: float, query_start_loc=None, max_q_len: int = 1, num_blocks=None,
           k_scale=None, v_scale=None, k_zp=None, v_zp=None, partition_size: int = 0,
           workspace=None, stream=None) -> None:
    """pa_decode; out/q [num_q_tokens, H, d]; caches [num_blocks, H_kv, 16, d]."""
    num_seqs = int(context_lens.shape[0])
    nq = int(q.shape[0])
    nb = k_cache.shape[0] if num_blocks is None else num_blocks
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_decode(_ptr(out), _dtype_code(out), _ptr(q), _dtype_code(q), _ptr(k_cache),
                           _ptr(v_cache), _dtype_code(k_cache), _ptr(k_scale), _ptr(v_scale),
                           _ptr(k_zp), _ptr(v_zp), _ptr(block_tables), block_tables.shape[1],
                           _ptr(context_lens), _ptr(query_start_loc), num_seqs, nq,
                           max_q_len if query_start_loc is not None else 1, q.shape[1],
                           k_cache.shape[1], q.shape[2], k_cache.shape[2], nb, float(scale),
                           int(max_context_len), int(partition_size), _ptr(workspace), ws_bytes,
                           _stream(stream)))


def decode_shared_prefix_workspace_size(num_seqs: int, num_q_tokens: int, num_heads: int,
                                        num_kv_heads: int, head_dim: int, max_q_len: int,
                                        max_context_len: int, num_groups: int,
                                        max_group_q_len: int, max_prefix_len: int,
                                        max_blocks_per_seq: int) -> int:
    return int(lib().pa_decode_shared_prefix_workspace_size(
        num_seqs, num_q_tokens, num_heads, num_kv_heads, head_dim, max_q_len, max_context_len,
        num_groups, max_group_q_len, max_prefix_len, max_blocks_per_seq))


def decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens,
                         max_context_len: int, scale: float, group_start, prefix_len,
                         max_group_q_len: int, max_prefix_len: int, query_start_loc=None,
                         max_q_len: int = 1, num_blocks=None, workspace=None,
                         stream=None) -> None:
    """pa_decode_shared_prefix; group_start / prefix_len: device int32 (see
    Pool.prefix_groups); other arguments as decode()."""
    num_seqs = int(context_lens.shape[0])
    nb = k_cache.shape[0] if num_blocks is None else num_blocks
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_shared_prefix(
        _ptr(out), _dtype_code(out), _ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache),
        _dtype_code(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
        _ptr(query_start_loc), num_seqs, int(q.shape[0]),
        max_q_len if query_start_loc is not None else 1, q.shape[1], k_cache.shape[1],
        q.shape[2], k_cache.shape[2], nb, float(scale), int(max_context_len), _ptr(group_start),
        _ptr(prefix_len), int(prefix_len.shape[0]), int(max_group_q_len), int(max_prefix_len),
        _ptr(workspace), ws_bytes, _stream(stream)))


NO_ALLOC_WORKSPACE_BYTES = 40 << 20
# Arrival counters at the start of every decode workspace (three regions of
# one uint32 per worker, 2048 workers at most): zero before a buffer's first
# call, left zero by every call.
ARRIVAL_BYTES = 3 * 4 * 2048


def decode_no_alloc(out, q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                    scale: float, query_start_loc=None, max_q_len: int = 1, num_blocks=None,
                    k_scale=None, v_scale=None, k_zp=None, v_zp=None, partition_size: int = 0,
                    stream=None) -> None:
    """pa_decode_no_alloc: decode with the library's built-in split-KV scratch
    (for callers that cannot allocate device memory); same arguments as
    decode() minus the workspace."""
    num_seqs = int(context_lens.shape[0])
    nb = k_cache.shape[0] if num_blocks is None else num_blocks
    _check(lib().pa_decode_no_alloc(
        _ptr(out), _dtype_code(out), _ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache),
        _dtype_code(k_cache), _ptr(k_scale), _ptr(v_scale), _ptr(k_zp), _ptr(v_zp),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), _ptr(query_start_loc),
        num_seqs, int(q.shape[0]), max_q_len if query_start_loc is not None else 1, q.shape[1],
        k_cache.shape[1], q.shape[2], k_cache.shape[2], nb, float(scale), int(max_context_len),
        int(partition_size), _stream(stream)))


# Bits of the device error word (PA_DEVERR_* in pa.h).
DEVERR_WAIT_FULL = 1 << 0      # a consumer gave up waiting for a staged tile
DEVERR_WAIT_EMPTY = 1 << 1     # a producer gave up waiting for a free stage
DEVERR_WAIT_DRAIN = 1 << 2     # the exit drain gave up on an in-flight copy
DEVERR_BAD_BLOCK = 1 << 3      # a block-table entry outside the pool
DEVERR_BAD_SLOT = 1 << 4       # a slot_mapping entry outside the pool
DEVERR_BAD_GROUP = 1 << 5      # a shared-prefix group range or prefix length
DEVERR_WORKSPACE = 1 << 6      # a workspace arrival counter was not zero


def device_error(stream=None) -> int:
    """pa_device_error: read and clear the device error word (synchronises);
    the value is a mask of the DEVERR_* bits."""
    code = ctypes.c_uint32()
    st = lib().pa_device_error(_stream(stream), ctypes.addressof(code))
    if st not in (0, 7):
        _check(st)
    return code.value

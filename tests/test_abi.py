"""The C-ABI library on the CPU: it loads, exports every symbol include/pa.h
declares, its host block pool agrees with the oracle's model operation by
operation, and argument errors are caught on the host before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_cache_154_gb300 as pa
from oracle.allocator import BlockPool, OutOfBlocks

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_154_gb300 import build
    build.build()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert len(names) >= 17
    L = ctypes.CDLL(pa.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert "sm_103a" in pa.version()


def test_device_error_bits_match_the_header():
    """The binding's DEVERR_* constants are the header's PA_DEVERR_* bits."""
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "pa.h")).read()
    bits = {m.group(1): 1 << int(m.group(2)) for m in
            re.finditer(r"#define PA_DEVERR_(\w+)\s+\(1u << (\d+)\)", hdr)}
    assert len(bits) == 7 and len(set(bits.values())) == 7
    for name, value in bits.items():
        assert getattr(pa, "DEVERR_" + name) == value, name


def test_pool_matches_oracle_model_on_random_ops():
    rng = np.random.default_rng(3)
    order = rng.permutation(300).astype(np.int32)
    c = pa.Pool(300, 16, order)
    m = BlockPool(300, 16, order)
    live = []
    for step in range(4000):
        op = int(rng.integers(0, 4))
        if op == 0 or not live:
            a, b = c.seq_create(), m.create()
            assert a == b
            live.append(a)
        elif op == 1:
            p = live[int(rng.integers(len(live)))]
            a, b = c.seq_fork(p), m.fork(p)
            assert a == b
            live.append(a)
        elif op == 2:
            s = live[int(rng.integers(len(live)))]
            n = int(rng.integers(0, 50))
            try:
                ms, mp = m.append_slots(s, n)
            except OutOfBlocks:
                with pytest.raises(pa.PAError) as e:
                    c.seq_append_slots(s, n)
                assert e.value.status == 3
                victim = live.pop(0)
                c.seq_free(victim)
                m.release(victim)
                continue
            cs, cp = c.seq_append_slots(s, n)
            assert cs.tolist() == ms and cp == mp
        else:
            s = live.pop(int(rng.integers(len(live))))
            c.seq_free(s)
            m.release(s)
        if step % 97 == 0 and live:
            mb = max(1, max(len(m.block_table(s)) for s in live))
            tables, lens = c.block_tables(live, mb)
            for i, s in enumerate(live):
                t = m.block_table(s)
                assert tables[i, :len(t)].tolist() == t and (tables[i, len(t):] == -1).all()
                assert lens[i] == m.lens[s]
            assert c.stats() == m.stats()
            for b in range(0, 300, 7):
                assert c.refcount(b) == m.ref[b]


def test_batched_reservations_match_the_model_step_by_step():
    """pa_seq_append_slots_batch against the allocator model on decode steps
    of forked sequences (every fork's first append into a shared tail block
    copies it): slots in sequence order, the copy-on-write pairs in order,
    the same state as one reservation per sequence; a step that runs out of
    blocks keeps the reservations before the failing sequence."""
    rng = np.random.default_rng(5)
    for trial in range(20):
        order = rng.permutation(200).astype(np.int32)
        c = pa.Pool(200, 16, order)
        m = BlockPool(200, 16, order)
        seqs = []
        for g in range(int(rng.integers(1, 5))):
            root = c.seq_create()
            assert m.create() == root
            n0 = int(rng.integers(1, 60))
            c.seq_append_slots(root, n0)
            m.append_slots(root, n0)
            seqs.append(root)
            for f in range(int(rng.integers(0, 4))):
                a = c.seq_fork(root)
                assert m.fork(root) == a
                seqs.append(a)
        for step in range(12):
            counts = rng.integers(0, 6, size=len(seqs)).astype(np.int32)
            want_slots, want_pairs, failed = [], [], None
            for i, (s, r) in enumerate(zip(seqs, counts)):
                try:
                    ms, mp = m.append_slots(s, int(r))
                except OutOfBlocks:
                    failed = i
                    break
                want_slots += ms
                if mp is not None:
                    want_pairs.append(list(mp))
            if failed is not None:
                with pytest.raises(pa.PAError) as e:
                    c.seq_append_slots_batch(seqs, counts)
                assert e.value.status == 3
                break
            got_slots, got_pairs = c.seq_append_slots_batch(seqs, counts)
            assert got_slots.tolist() == want_slots
            assert got_pairs.tolist() == want_pairs
            tables, lens = c.block_tables(seqs, 64)
            for i, s in enumerate(seqs):
                t = m.block_table(s)
                assert tables[i, :len(t)].tolist() == t and lens[i] == m.lens[s]
            assert c.stats() == m.stats()
    # state after a failing step: the sequences before the failing one were reserved
    c = pa.Pool(4, 16, np.arange(4, dtype=np.int32))
    a, b = c.seq_create(), c.seq_create()
    with pytest.raises(pa.PAError):
        c.seq_append_slots_batch([a, b], [48, 48])      # 3 blocks, then 3 more of 4
    assert c.seq_len(a) == 48 and c.seq_len(b) == 0


def test_pool_errors():
    with pytest.raises(pa.PAError) as e:
        pa.Pool(8, 32)
    assert e.value.status == 2                           # block size other than 16
    with pytest.raises(pa.PAError):
        pa.Pool(4, 16, [0, 1, 1, 2])                     # not a permutation
    p = pa.Pool(4, 16)
    s = p.seq_create()
    with pytest.raises(pa.PAError) as e:
        p.seq_append_slots(s, 65)
    assert e.value.status == 3 and p.seq_len(s) == 0 and p.stats() == (4, 0, 0)
    p.seq_free(s)
    with pytest.raises(pa.PAError) as e:
        p.seq_free(s)                                    # double free
    assert e.value.status == 1
    with pytest.raises(pa.PAError):
        p.seq_fork(99)


def test_device_calls_reject_bad_arguments_on_the_host():
    L = pa.lib()
    # NULL pointers, unsupported head_dim / block_size: nothing is launched
    st = L.pa_decode(None, 2, None, 1, None, None, 1, None, None, None, None, None, 4, None,
                     None, 2, 2, 1, 8, 2, 128, 16, 10, 0.1, 64, 0, None, 0, None)
    assert st == 1
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf)
    st = L.pa_decode(p, 2, p, 1, p, p, 1, None, None, None, None, p, 4, p, None, 2, 2, 1, 8,
                     2, 96, 16, 10, 0.1, 64, 0, None, 0, None)
    assert st == 2 and b"head_dim" in L.pa_last_error()
    st = L.pa_decode(p, 2, p, 1, p, p, 1, None, None, None, None, p, 4, p, None, 2, 2, 1, 8,
                     3, 128, 16, 10, 0.1, 64, 0, None, 0, None)
    assert st == 1                                       # 8 heads over 3 KV heads
    st = L.pa_decode(p, 2, p, 0, p, p, 1, None, None, None, None, p, 4, p, None, 2, 2, 1, 8,
                     2, 128, 16, 10, 0.1, 64, 0, None, 0, None)
    assert st == 2                                       # q fp16 against a bf16 cache
    st = L.pa_decode(p, 2, p, 1, p, p, 1, None, None, None, None, p, 4, p, None, 2, 2, 1, 8,
                     2, 128, 16, 10, 0.1, 4096, 0, None, 0, None)
    assert st == 1 and b"max_blocks" in L.pa_last_error()   # table too narrow
    st = L.pa_decode(p, 2, p, 1, p, p, 1, None, None, None, None, p, 512, p, None, 2, 2, 1, 8,
                     2, 128, 16, 10, 0.1, 4096, 0, None, 0, None)
    assert st == 1 and b"workspace" in L.pa_last_error()    # balanced schedule needs one
    st = L.pa_decode(p, 2, p, 1, p, p, 1, None, None, None, None, p, 512, p, None, 2, 2, 1, 8,
                     2, 128, 16, 10, 0.1, 4096, 24, None, 0, None)
    assert st == 1 and b"partition_size" in L.pa_last_error()   # not a multiple of 16
    st = L.pa_append_kv(p, p, 1, p, p, 0, None, None, None, None, p, 3, 10, 2, 128, 16, None)
    assert st == 2                                       # bf16 rows into an fp16 cache
    st = L.pa_append_kv(p, p, 1, p, p, 3, None, None, None, None, p, 3, 10, 2, 128, 16, None)
    assert st == 1                                       # INT8 cache without scales
    st = L.pa_copy_blocks(p, p, None, None, None, None, p, 1, 10, 2, 128, 8, 1, None)
    assert st == 2                                       # block_size 8
    assert L.pa_copy_blocks(None, None, None, None, None, None, None, 0, 10, 2, 128, 16, 1,
                            None) == 0                   # nothing to copy


def test_workspace_size():
    # every workspace starts with 6144 uint32 arrival counters (24576 bytes)
    arr = 24576
    assert arr == pa.ARRIVAL_BYTES
    # partitioned schedule: o, m, l per (q token, head, partition)
    assert pa.decode_workspace_size(64, 64, 32, 8, 128, 1, 512, 512) == 0
    n = pa.decode_workspace_size(4, 4, 32, 8, 128, 1, 131072, 512)
    rows = 4 * 32 * 256
    assert n == arr + rows * 128 * 4 + 2 * rows * 4
    # balanced schedule: prefix sums, then 2 slots per worker (workers capped at 2048);
    # a slot is a 32-byte header + m, l, O for a tile of 16 (or 64) query rows
    slot = 32 + 4 * 16 * (128 + 2)
    assert pa.decode_workspace_size(64, 64, 32, 8, 128, 1, 4096, 0) == \
        arr + 512 + 2 * 2048 * slot
    slot64 = 32 + 4 * 16 * 66
    assert pa.decode_workspace_size(1, 1, 8, 2, 64, 1, 17, 0) == arr + 256 + 2 * (2 * 2) * slot64
    # 32 q heads on one KV head with verify runs of 5 (160 rows): slots sized for the
    # 64-row tiles of the 16-bit kernels (the INT8 and FP8 kernels use 16-row tiles)
    slot_big = 32 + 4 * 64 * 130
    assert pa.decode_workspace_size(256, 400, 32, 1, 128, 5, 16384, 0) == \
        arr + 1280 + 2 * 2048 * slot_big
    assert pa.decode_workspace_size(1, 1, 8, 3, 64, 1, 17, 0) == 0      # heads not a multiple


def test_prefix_groups_match_model_on_fork_trees():
    """pa_pool_prefix_groups against the allocator model on random fork
    trees (forks listed next to their prompt), with query runs of 1-5."""
    rng = np.random.default_rng(11)
    for trial in range(40):
        order = rng.permutation(400).astype(np.int32)
        c = pa.Pool(400, 16, order)
        m = BlockPool(400, 16, order)
        seqs = []
        for g in range(int(rng.integers(1, 5))):
            root = c.seq_create()
            assert m.create() == root
            n = int(rng.integers(1, 120))
            c.seq_append_slots(root, n)
            m.append_slots(root, n)
            members = [root]
            for _ in range(int(rng.integers(0, 5))):
                parent = members[int(rng.integers(len(members)))]
                child = c.seq_fork(parent)
                assert m.fork(parent) == child
                members.append(child)
            for s in members:
                k = int(rng.integers(0, 40))
                c.seq_append_slots(s, k)
                m.append_slots(s, k)
            seqs += members
        q_lens = [int(rng.integers(1, min(5, m.lens[s]) + 1)) for s in seqs]
        gs, pl = c.prefix_groups(seqs, q_lens)
        mgs, mpl = m.prefix_groups(seqs, q_lens)
        assert gs.tolist() == mgs and pl.tolist() == mpl
        # what a prefix promises: shared physical blocks, before every query
        for g in range(len(pl)):
            members = seqs[gs[g]:gs[g + 1]]
            nb = pl[g] // 16
            assert pl[g] % 16 == 0
            for i, s in zip(range(gs[g], gs[g + 1]), members):
                assert m.block_table(s)[:nb] == m.block_table(members[0])[:nb]
                assert pl[g] <= m.lens[s] - q_lens[i] + 1
    with pytest.raises(pa.PAError):
        c.prefix_groups([9999])


def _trace_ops(rng, n_ops, prompts):
    """A serving-like trace: requests share system prompts (page 1 §2.4's
    example) and differ after them; some finish, some get forked."""
    ops = []
    for _ in range(n_ops):
        u = rng.random()
        if u < 0.45:
            p = prompts[int(rng.integers(len(prompts)))]
            user = rng.integers(0, 50, size=int(rng.integers(1, 40))).tolist()
            ops.append(("req", p + user))
        elif u < 0.65:
            ops.append(("gen", int(rng.integers(1, 20))))
        elif u < 0.75:
            ops.append(("fork", None))
        elif u < 0.80:
            ops.append(("plain", int(rng.integers(1, 20))))
        else:
            ops.append(("free", None))
    return ops


@pytest.mark.parametrize("max_cached", [0, 8, 64])
def test_prefix_cache_matches_model_on_serving_traces(max_cached):
    rng = np.random.default_rng(17 + max_cached)
    prompts = [rng.integers(0, 50, size=n).tolist() for n in (200, 64, 37, 16, 5)]
    order = rng.permutation(180).astype(np.int32)
    c = pa.Pool(180, 16, order)
    m = BlockPool(180, 16, order)
    c.enable_prefix_cache(max_cached)
    m.enable_prefix_cache(max_cached)
    live = []
    for kind, arg in _trace_ops(rng, 1500, prompts):
        try:
            if kind == "req":
                ms, mn = m.create_with_prefix(arg)
                cs, cn = c.create_with_prefix(arg)
                assert (cs, cn) == (ms, mn)
                live.append(ms)
                try:
                    mslots, mp = m.append_tokens(ms, arg[mn:])
                except OutOfBlocks:
                    with pytest.raises(pa.PAError):
                        c.append_tokens(cs, arg[cn:])
                    raise
                cslots, cp = c.append_tokens(cs, arg[cn:])
                assert cslots.tolist() == mslots and cp == mp
            elif kind == "gen" and live:
                s = live[int(rng.integers(len(live)))]
                toks = rng.integers(0, 50, size=arg).tolist()
                try:
                    mslots, mp = m.append_tokens(s, toks)
                except OutOfBlocks:
                    with pytest.raises(pa.PAError):
                        c.append_tokens(s, toks)
                    raise
                cslots, cp = c.append_tokens(s, toks)
                assert cslots.tolist() == mslots and cp == mp
            elif kind == "plain" and live:
                s = live[int(rng.integers(len(live)))]
                try:
                    mslots, mp = m.append_slots(s, arg)
                except OutOfBlocks:
                    with pytest.raises(pa.PAError):
                        c.seq_append_slots(s, arg)
                    raise
                cslots, cp = c.seq_append_slots(s, arg)
                assert cslots.tolist() == mslots and cp == mp
            elif kind == "fork" and live:
                p = live[int(rng.integers(len(live)))]
                assert c.seq_fork(p) == m.fork(p)
                live.append(m._next - 1)
            elif kind == "free" and live:
                s = live.pop(int(rng.integers(len(live))))
                c.seq_free(s)
                m.release(s)
        except OutOfBlocks:
            while len(live) > 3:                 # make room, then carry on
                s = live.pop(0)
                c.seq_free(s)
                m.release(s)
        assert c.stats() == m.stats()
        assert c.prefix_stats() == m.prefix_stats()
    for s in live:
        mb = max(1, len(m.block_table(s)))
        t, l = c.block_tables([s], mb)
        assert t[0, :len(m.block_table(s))].tolist() == m.block_table(s)
    assert m.hits > 50                           # the trace really reuses prefixes


def test_prefix_cache_api_errors():
    c = pa.Pool(8, 16)
    with pytest.raises(pa.PAError):
        c.create_with_prefix([1, 2, 3])          # not enabled
    s = c.seq_create()
    with pytest.raises(pa.PAError):
        c.append_tokens(s, [1])
    with pytest.raises(pa.PAError):
        c.enable_prefix_cache(-1)

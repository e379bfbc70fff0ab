"""Pins for the block-pool model, the KV-size formula, append and block copy
(CPU only). Sources: page 3 (devpress.csdn.net) §七 block tables and
KVBlockManager; page 1 §2.3 waste bound; page 2 (ybb.press) §2.1 best-of-N
saving; page 4 (cs336 lecture 10) KV-size table."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle.allocator import BlockPool, OutOfBlocks
from oracle import formulas

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_page3_worked_block_tables():
    g = json.load(open(os.path.join(GOLD, "block_table_p3.json")))
    bs = g["block_size"]
    A, B = g["tables"]["A"], g["tables"]["B"]
    # free list popped from its end: arrange it so the pops give the page's tables
    rest = [b for b in range(32) if b not in A + B]
    pool = BlockPool(32, bs, rest + list(reversed(B)) + list(reversed(A)))
    a = pool.create()
    pool.append_slots(a, 4 * bs)
    b = pool.create()
    pool.append_slots(b, 3 * bs - 5)
    assert pool.block_table(a) == A and pool.block_table(b) == B
    for logical, phys in g["logical_to_physical"]:
        assert pool.block_table(a)[logical] == phys
    # slot of token 20 of A: logical block 1 -> physical 4, offset 4
    pool2 = BlockPool(32, bs, rest + list(reversed(B)) + list(reversed(A)))
    s = pool2.create()
    slots, _ = pool2.append_slots(s, 21)
    assert slots[20] == 4 * bs + 4


def test_page3_manager_semantics():
    bs = 16
    pool = BlockPool(10, bs)
    s = pool.create()
    slots, pair = pool.append_slots(s, 33)           # ceil(33/16) = 3 blocks
    assert len(pool.block_table(s)) == 3 and pair is None
    assert pool.block_table(s) == [9, 8, 7]          # list(range(n)).pop() order
    # a new block is taken exactly when used == capacity
    pool.append_slots(s, 14)                          # 47 tokens: still 3 blocks
    assert len(pool.block_table(s)) == 3
    pool.append_slots(s, 1)                           # 48: full, still 3
    assert len(pool.block_table(s)) == 3
    pool.append_slots(s, 1)                           # 49th token needs block 4
    assert len(pool.block_table(s)) == 4
    # shortage raises and changes nothing
    t = pool.create()
    before = (list(pool.free), list(pool.ref))
    with pytest.raises(OutOfBlocks):
        pool.append_slots(t, 7 * bs)
    assert (list(pool.free), list(pool.ref)) == before and pool.lens[t] == 0
    # release returns all blocks
    pool.release(s)
    assert sorted(pool.free) == list(range(10))


def test_fork_and_copy_on_write():
    pool = BlockPool(8, 16)
    p = pool.create()
    pool.append_slots(p, 20)                           # 2 blocks, tail partial
    c = pool.fork(p)
    assert pool.block_table(c) == pool.block_table(p)
    assert all(pool.ref[b] == 2 for b in pool.block_table(p))
    slots, pair = pool.append_slots(c, 1)              # writes into the shared tail -> copy
    assert pair is not None and pair[0] == pool.block_table(p)[1]
    assert pool.block_table(c)[1] == pair[1] and pool.block_table(c)[0] == pool.block_table(p)[0]
    assert slots == [pair[1] * 16 + 4]
    assert pool.ref[pair[0]] == 1 and pool.ref[pair[1]] == 1
    # the parent is now sole owner of its tail: writes in place
    slots, pair2 = pool.append_slots(p, 1)
    assert pair2 is None and slots == [pool.block_table(p)[1] * 16 + 4]
    # a full shared tail needs no copy: the next token opens a fresh block
    q = pool.create()
    pool.append_slots(q, 16)
    r = pool.fork(q)
    _, pair3 = pool.append_slots(r, 1)
    assert pair3 is None and pool.block_table(r)[0] == pool.block_table(q)[0]


def test_random_ops_keep_refcounts_consistent():
    rng = np.random.default_rng(7)
    pool = BlockPool(200, 16, rng.permutation(200))
    live = []
    for _ in range(3000):
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                live.append(pool.create())
            elif op == 1:
                live.append(pool.fork(live[rng.integers(len(live))]))
            elif op == 2:
                s = live[rng.integers(len(live))]
                slots, pair = pool.append_slots(s, int(rng.integers(1, 40)))
                for x in slots:                       # every written slot is unshared
                    assert pool.ref[x // 16] == 1
            else:
                pool.release(live.pop(rng.integers(len(live))))
        except OutOfBlocks:
            pool.release(live.pop(0))
        # conservation: sum of refcounts == total table entries; free + used == all
        assert sum(pool.ref) == sum(len(pool.block_table(s)) for s in live)
        free, used, _ = pool.stats()
        assert free + used == 200 and not (set(pool.free) & {b for b in range(200) if pool.ref[b]})
        for s in live:                                   # waste below one block (page 1 §2.3)
            assert len(pool.block_table(s)) == math.ceil(pool.lens[s] / 16)


def test_best_of_5_saves_over_75_percent():
    wl = W.llama2_70b_best_of_5()
    run = oracle.run(wl, decode=False)
    free, used, shared = run.pool.stats()
    unshared = sum(math.ceil(L / 16) for L in run.context_lens)
    saving = 1 - used / unshared
    assert saving > 0.75, saving                          # page 2 §2.1: N=5 saves > 75%
    assert len(run.step_pairs) >= 8                       # the step copies each group's tail


def test_kv_formula_matches_page4_table():
    g = json.load(open(os.path.join(GOLD, "kv_size_p4.json")))
    for row in g["rows"]:
        b = formulas.kv_cache_bytes_dmodel(row["layers"], row["d_model"], row["seq_len"],
                                           row["dtype_bytes"])
        assert b / 1024 ** 3 == row["size"], row
        # the heads x head_dim form agrees (MHA: 32 heads of 128, 64 heads of 128)
        heads = row["d_model"] // 128
        assert formulas.kv_cache_bytes(row["layers"], heads, 128, row["seq_len"], 1,
                                       row["dtype_bytes"]) == b


def test_kv_formula_equals_bytes_allocated():
    # pool blocks x bytes per block == formula when every length is a multiple of 16;
    # ragged lengths round each sequence up by less than one block
    for lens in ([16, 64, 4096], [17, 33, 64, 100]):
        wl = W.simple("f", 3, lens, [1] * len(lens), 8, 2, 64, "f16", pool_factor=1.0)
        run = oracle.run(wl, decode=False)
        _, used, _ = run.pool.stats()
        per_block = 2 * wl.num_kv_heads * 16 * wl.head_dim * 2
        allocated = used * per_block
        assert allocated == formulas.paged_bytes(1, 2, 64, lens, 2)
        exact = formulas.kv_cache_bytes(1, 2, 64, sum(lens), 1, 2)
        assert 0 <= allocated - exact < len(lens) * per_block
        if all(L % 16 == 0 for L in lens):
            assert allocated == exact


def test_append_then_gather_round_trips_and_spares_canaries():
    wl = W.simple("rt", 5, [17, 33, 64, 100], [1, 2, 1, 3], 8, 2, 64, "bf16")
    run = oracle.run(wl, canary_blocks=W.CANARY_BLOCKS, canary_byte=W.CANARY_BYTE)
    c = run.cache
    for s, (K, V) in enumerate(W.contiguous_kv(wl)):
        L = K.shape[0]
        t = np.arange(L)
        blk = run.block_tables[s, t // 16]
        got_k = c.k[blk, :, t % 16, :]
        want = K.view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got_k, want)
        assert np.array_equal(c.v[blk, :, t % 16, :], V.view(torch.int16).numpy().view(np.uint16))
    assert (c.k[wl.num_blocks:].view(np.uint8) == W.CANARY_BYTE).all()
    # negative slots are skipped
    k2 = oracle.empty_cache("bf16", 4, 2, 16, 64)
    oracle.append(k2, wl.step[0].k, wl.step[0].v, np.array([-1]), "bf16")
    assert not k2.k.any()


def test_copy_blocks_copies_whole_blocks_only():
    c = oracle.empty_cache("int8", 6, 2, 16, 64)
    rng = np.random.default_rng(0)
    for a in c.arrays():
        a.view(np.uint8)[...] = rng.integers(0, 256, a.nbytes, dtype=np.uint8).reshape(a.view(np.uint8).shape)
    before = [a.copy().view(np.uint8) for a in c.arrays()]
    oracle.copy_blocks(c, [(1, 4), (2, 0)])
    for a, b in zip([x.view(np.uint8) for x in c.arrays()], before):
        assert np.array_equal(a[4], b[1]) and np.array_equal(a[0], b[2])
        for blk in (1, 2, 3, 5):
            assert np.array_equal(a[blk], b[blk])


def test_prefix_groups_model_is_maximal_and_sound():
    """The model's prefix is the longest whole-block prefix that every fork
    holds in the same physical blocks and that precedes every query: one
    block more breaks one of those conditions."""
    pool = BlockPool(200, 16)
    root = pool.create()
    pool.append_slots(root, 70)                  # 4 full blocks + 6 tokens
    a = pool.fork(root)
    b = pool.fork(root)
    pool.append_slots(a, 3)                      # CoW of the shared tail block
    pool.append_slots(b, 30)
    lone = pool.create()
    pool.append_slots(lone, 40)
    gs, pl = pool.prefix_groups([root, a, b, lone])
    assert gs == [0, 3, 4] and pl == [64, 0]     # 4 shared full blocks; a group of one gets 0
    # a query run that reaches into the 4th block caps the prefix at 3 blocks
    gs, pl = pool.prefix_groups([root, a, b], q_lens=[1, 1, 70 + 30 - 63 + 1])
    assert pl == [48]
    # forks that are not adjacent form separate groups
    gs, pl = pool.prefix_groups([root, lone, a])
    assert gs == [0, 1, 2, 3] and pl == [0, 0, 0]


def test_prefix_cache_model_reuses_exactly_the_same_prefixes():
    """What the model promises: a reused block holds the very tokens the new
    request starts with (the whole prefix up to that block, not just the
    block's own 16 tokens), at least one token is left to compute, and a
    different earlier token breaks the chain even when later blocks agree."""
    pool = BlockPool(64, 16)
    pool.enable_prefix_cache(16)
    toks = list(range(100, 150))                     # 50 tokens: 3 full blocks + 2
    a = pool.create()
    pool.append_tokens(a, toks)
    assert pool.prefix_stats()[1] == 3               # three full blocks registered
    b, n = pool.create_with_prefix(toks + [7])
    assert n == 48 and pool.block_table(b) == pool.block_table(a)[:3]
    c, n = pool.create_with_prefix(toks[:48])        # exactly 3 blocks: keep one token
    assert n == 32
    d, n = pool.create_with_prefix([0] + toks[1:])   # first token differs
    assert n == 0
    e, n = pool.create_with_prefix(toks[:16] + [9] * 16 + toks[32:] + [1])
    assert n == 16                                   # block 1 differs, block 2 unreachable
    for s in (a, b, c, d, e):
        pool.release(s)
    assert pool.prefix_stats()[0] == 3               # registered blocks wait in the LRU


def test_prefix_cache_model_lru_eviction_order():
    """Released registered blocks leave in the order they were released
    (oldest first) once the LRU is over capacity, and allocation takes the
    free list before evicting anything."""
    pool = BlockPool(6, 16, free_order=range(6))
    pool.enable_prefix_cache(2)
    seqs = []
    for base in (0, 1000, 2000):
        s = pool.create()
        pool.append_tokens(s, list(range(base, base + 16)))   # one full block each
        seqs.append(s)
    blocks = [pool.block_table(s)[0] for s in seqs]
    for s in seqs:
        pool.release(s)
    assert list(pool.lru) == blocks[1:]              # capacity 2: the first was evicted
    assert pool.free[-1] == blocks[0]
    s, n = pool.create_with_prefix(list(range(1000, 1016)) + [5])
    assert n == 16 and list(pool.lru) == blocks[2:]  # a hit revives its block
    t = pool.create()
    assert len(pool.free) == 4
    pool.append_slots(t, 16 * 4)                     # the four free blocks: no eviction
    assert list(pool.lru) == blocks[2:]
    pool.append_slots(t, 16)                         # free list empty: evict the oldest
    assert list(pool.lru) == [] and pool.prefix_stats()[1] == 1

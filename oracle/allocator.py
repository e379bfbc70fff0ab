"""Block-pool model -- the oracle for block allocation, forks and copy-on-write.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and
bench.py's CPU-baseline leg, never by the CUDA library or its binding.

It restates the block manager sketched on page 3 ("KV Cache ... PagedAttention",
devpress.csdn.net, §七 "PagedAttention 如何解决显存碎片"):

* a free list that starts as the given order (the page uses range(n)) and is
  popped from its end;
* a sequence of n tokens holds ceil(n / block_size) blocks, and a new block is
  taken exactly when the token count reaches the capacity (used >= capacity);
* running out of free blocks is an error;
* releasing a sequence returns its blocks to the end of the free list.

and adds what that section lists as missing from its sketch (block reference
counts, prefix sharing, copy-on-write), as page 2 ("ybb.press" §2.1, best-of-N
sharing that copies a block only when it is modified) describes:

* fork(parent) gives the child the parent's block table and raises the
  reference count of every block in it;
* appending into a partially filled tail block whose reference count is above
  one first takes a fresh block, records the pair (old, fresh) as a block copy,
  moves this sequence's table entry to the fresh block and lowers the old
  block's count. The copy block is taken before any new tail blocks;
* release lowers every count and frees the blocks that reach zero, in table
  order.

An append is all-or-nothing: if the free list cannot cover it, nothing changes.
"""
from __future__ import annotations

from collections import OrderedDict
from typing import Dict, List, Optional, Sequence, Tuple


class OutOfBlocks(RuntimeError):
    pass


class BadSequence(KeyError):
    pass


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int = 16,
                 free_order: Optional[Sequence[int]] = None):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad pool shape")
        self.num_blocks = num_blocks
        self.block_size = block_size
        if free_order is None:
            free_order = range(num_blocks)
        self.free: List[int] = [int(b) for b in free_order]
        if sorted(self.free) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self.ref: List[int] = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        self._next = 0
        # prefix cache (see enable_prefix_cache)
        self.pc_on = False
        self.pc_max = 0
        self.nodes: Dict[int, list] = {}          # id -> [parent, tokens, block, children]
        self.edges: Dict[tuple, int] = {}         # (parent, tokens) -> id
        self.next_node = 0
        self.block_node: Dict[int, int] = {}      # registered block -> node
        self.lru: "OrderedDict[int, None]" = OrderedDict()   # oldest first
        self.seq_nodes: Dict[int, List[int]] = {}
        self.seq_tail: Dict[int, List[int]] = {}
        self.seq_known: Dict[int, bool] = {}
        self.hits = 0
        self.lookups = 0

    # -- sequences ---------------------------------------------------------
    def create(self) -> int:
        sid = self._next
        self._next += 1
        self.tables[sid] = []
        self.lens[sid] = 0
        self.seq_nodes[sid] = []
        self.seq_tail[sid] = []
        self.seq_known[sid] = True
        return sid

    def _get(self, sid: int) -> List[int]:
        if sid not in self.tables:
            raise BadSequence(sid)
        return self.tables[sid]

    def fork(self, parent: int) -> int:
        table = self._get(parent)
        child = self.create()
        self.tables[child] = list(table)
        self.lens[child] = self.lens[parent]
        self.seq_nodes[child] = list(self.seq_nodes[parent])
        self.seq_tail[child] = list(self.seq_tail[parent])
        self.seq_known[child] = self.seq_known[parent]
        for b in table:
            self.ref[b] += 1
        return child

    def append_slots(self, sid: int, n: int) -> Tuple[List[int], Optional[Tuple[int, int]]]:
        """Reserve n token slots; returns (slots, copy pair or None)."""
        table = self._get(sid)
        if n < 0:
            raise ValueError("n < 0")
        bs = self.block_size
        L = self.lens[sid]
        if n == 0:
            return [], None
        cow = (L % bs != 0) and self.ref[table[-1]] > 1
        new_blocks = -(-(L + n) // bs) - len(table)
        avail = len(self.free) + len(self.lru)
        if new_blocks + (1 if cow else 0) > avail:
            raise OutOfBlocks(f"need {new_blocks + int(cow)} blocks, {avail} free")
        pair = None
        if cow:
            src = table[-1]
            dst = self._take()
            self.ref[src] -= 1
            self.ref[dst] = 1
            table[-1] = dst
            pair = (src, dst)
        slots = []
        for i in range(n):
            pos = L + i
            if pos >= len(table) * bs:
                b = self._take()
                self.ref[b] = 1
                table.append(b)
            slots.append(table[pos // bs] * bs + pos % bs)
        self.lens[sid] = L + n
        if n > 0 and not self._with_tokens:
            self.seq_known[sid] = False          # tokens unknown: nothing more to register
        return slots, pair

    _with_tokens = False

    def release(self, sid: int) -> None:
        table = self._get(sid)
        for b in table:
            if self.ref[b] <= 0:
                raise RuntimeError(f"refcount underflow on block {b}")
        for b in table:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self._release(b)
        del self.tables[sid]
        del self.lens[sid]
        del self.seq_nodes[sid]
        del self.seq_tail[sid]
        del self.seq_known[sid]

    # -- views -------------------------------------------------------------
    def block_table(self, sid: int) -> List[int]:
        return list(self._get(sid))

    def stats(self) -> Tuple[int, int, int]:
        used = sum(1 for r in self.ref if r > 0)
        shared = sum(1 for r in self.ref if r > 1)
        return len(self.free), used, shared

    def prefix_groups(self, seqs: Sequence[int],
                      q_lens: Optional[Sequence[int]] = None) -> Tuple[List[int], List[int]]:
        """Fork groups for read-once shared-prefix decode: runs of adjacent
        sequences (in the given order) whose first physical block is the same
        -- forks of one prompt (page 2 §2.1, best-of-N) -- and, per group, the
        tokens at the front that every member holds in the same physical
        blocks and that precede every member's first query: whole blocks
        only, at most (L - r + 1) // block_size of them for a member with L
        tokens and a query run of r. A group of one gets prefix 0.
        Returns (group_start [G + 1], prefix_len [G])."""
        bs = self.block_size
        seqs = [int(s) for s in seqs]
        rs = [1] * len(seqs) if q_lens is None else [int(r) for r in q_lens]
        for s, r in zip(seqs, rs):
            self._get(s)
            if not 1 <= r <= self.lens[s]:
                raise ValueError(f"sequence {s}: query run {r}")
        starts, prefixes = [], []
        i = 0
        while i < len(seqs):
            first = self.tables[seqs[i]]
            j = i + 1
            while (j < len(seqs) and first and self.tables[seqs[j]]
                   and self.tables[seqs[j]][0] == first[0]):
                j += 1
            k = 0
            if j - i > 1:
                members = range(i, j)
                # longest run of leading entries equal in every member's table
                k = min(len(self.tables[seqs[m]]) for m in members)
                for m in members:
                    t = self.tables[seqs[m]]
                    c = 0
                    while c < k and t[c] == first[c]:
                        c += 1
                    k = c
                # no prefix token may reach a member's first query
                k = min([k] + [(self.lens[seqs[m]] - rs[m] + 1) // bs for m in members])
            starts.append(i)
            prefixes.append(k * bs)
            i = j
        starts.append(len(seqs))
        return starts, prefixes

    # -- prefix cache ------------------------------------------------------
    # Page 1 ("大模型推理优化全攻略" §2.4) sketches a prefix KV cache: a hash of
    # the prefix tokens finds the cached KV, lookups refresh an entry, and an
    # ordered dict evicts the least recently used one past a capacity; page 3
    # states the mapping hash(prefix_tokens) -> KV blocks. Restated per block:
    # a full block is named by the whole token prefix ending with it, a trie
    # node (parent node, the block's tokens); blocks no sequence holds wait in
    # an LRU of at most max_cached_blocks, and allocation evicts its oldest
    # entry only when the free list is empty.

    def enable_prefix_cache(self, max_cached_blocks: int) -> None:
        if max_cached_blocks < 0:
            raise ValueError("max_cached_blocks < 0")
        self.pc_on = True
        self.pc_max = max_cached_blocks
        while len(self.lru) > self.pc_max:
            old, _ = self.lru.popitem(last=False)
            self._unregister(old)
            self.free.append(old)

    def _take(self) -> int:
        if self.free:
            return self.free.pop()
        b, _ = self.lru.popitem(last=False)
        self._unregister(b)
        return b

    def _release(self, b: int) -> None:
        if b not in self.block_node:
            self.free.append(b)
            return
        self.lru[b] = None
        if len(self.lru) > self.pc_max:
            old, _ = self.lru.popitem(last=False)
            self._unregister(old)
            self.free.append(old)

    def _unregister(self, b: int) -> None:
        nid = self.block_node.pop(b, None)
        if nid is None:
            return
        self.nodes[nid][2] = -1
        while nid >= 0 and nid in self.nodes:
            parent, tokens, block, children = self.nodes[nid]
            if block >= 0 or children > 0:
                return
            del self.edges[(parent, tokens)]
            del self.nodes[nid]
            if parent >= 0:
                self.nodes[parent][3] -= 1
            nid = parent

    def _node(self, parent: int, tokens: tuple) -> int:
        nid = self.edges.get((parent, tokens))
        if nid is None:
            nid = self.next_node
            self.next_node += 1
            self.nodes[nid] = [parent, tokens, -1, 0]
            self.edges[(parent, tokens)] = nid
            if parent >= 0:
                self.nodes[parent][3] += 1
        return nid

    def append_tokens(self, sid: int, tokens: Sequence[int]) -> Tuple[List[int], Optional[Tuple[int, int]]]:
        """append_slots for known token ids; every block this fills is
        registered under its prefix (unless that prefix already has a block)."""
        if not self.pc_on:
            raise ValueError("the prefix cache is not enabled")
        L = self.lens[sid] if sid in self.lens else 0
        self._with_tokens = True
        try:
            slots, pair = self.append_slots(sid, len(tokens))
        finally:
            self._with_tokens = False
        if not self.seq_known[sid]:
            return slots, pair
        bs = self.block_size
        tail, chain = self.seq_tail[sid], self.seq_nodes[sid]
        for i, t in enumerate(tokens):
            tail.append(int(t))
            if len(tail) < bs:
                continue
            b = (L + i) // bs
            parent = -1 if b == 0 else chain[b - 1]
            if parent >= 0 and parent not in self.nodes:
                self.seq_known[sid] = False
                break
            nid = self._node(parent, tuple(tail))
            chain.append(nid)
            blk = self.tables[sid][b]
            if self.nodes[nid][2] < 0 and blk not in self.block_node:
                self.nodes[nid][2] = blk
                self.block_node[blk] = nid
            tail.clear()
        return slots, pair

    def create_with_prefix(self, tokens: Sequence[int]) -> Tuple[int, int]:
        """A new sequence holding the longest chain of cached whole blocks
        that the tokens start with, leaving at least one token to compute.
        Returns (sequence id, tokens already cached)."""
        if not self.pc_on:
            raise ValueError("the prefix cache is not enabled")
        sid = self.create()
        bs = self.block_size
        parent = -1
        b = 0
        while (b + 1) * bs <= len(tokens) - 1:
            self.lookups += 1
            nid = self.edges.get((parent, tuple(int(t) for t in tokens[b * bs:(b + 1) * bs])))
            if nid is None or self.nodes[nid][2] < 0:
                break
            blk = self.nodes[nid][2]
            if self.ref[blk] == 0:
                del self.lru[blk]
            self.ref[blk] += 1
            self.tables[sid].append(blk)
            self.seq_nodes[sid].append(nid)
            self.hits += 1
            parent = nid
            b += 1
        self.lens[sid] = b * bs
        return sid, b * bs

    def prefix_stats(self) -> Tuple[int, int, int, int]:
        """(cached unreferenced blocks, registered blocks, hit blocks, looked-up blocks)."""
        return len(self.lru), len(self.block_node), self.hits, self.lookups


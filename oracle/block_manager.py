"""Block manager (free list, refcounts, fork, append with copy-on-write, free) — the oracle.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``): never imported by the library.

The rules, in the pages' order:

* A fixed pool of ``num_blocks`` physical blocks of ``block_size`` token slots
  is carved at start-up ("PagedAttention: How vLLM Borrowed Virtual Memory...",
  section "The OS-Inspired Insight", item 1; "PagedAttention and vLLM: Virtual
  Memory for the KV Cache", section "L2 — Mechanism", the block pool).
* Allocation pops a block off the free list, freeing pushes it back, both O(1)
  ("What is paged attention?", section "How it works").  The pages leave the
  order open ("say P0 and P1"); the oracle's free list is a LIFO stack whose
  first pops return ``pop_order`` in order (ascending ids by default).
* Each physical block carries a reference count of the logical blocks that
  point at it ("PagedAttention — how vLLM stopped wasting 80%...", section
  "Memory sharing: copy-on-write ..."); a block returns to the free list when
  its count reaches zero.
* ``fork`` gives a child a copy of the parent's block table and increments the
  count of every block in it (same section; "Walking Through the Lifecycle",
  Copy-on-Write).
* ``append`` writes tokens one position ``p`` at a time:
  - ``p % B == 0``: the last block is full (or the table is empty), so a new
    block is allocated and appended to the table — never a copy, even if the
    previous block is shared (worked example "three requests, one memory
    pool", step 3; "position modulo 16 equals 0", section "Walking Through
    the Lifecycle", Decode);
  - otherwise, if the last block's count is above one, the writer gets a
    private copy: allocate a new block, record the (old, new) copy pair,
    decrement the old block, and put the new block at the end of the table
    (section "Copy-on-Write for Beam Search and Parallel Sampling": "detects
    ref_count > 1, allocates a new physical block, copies the content,
    decrements the original's ref_count");
  - the token's slot is ``table[p // B] * B + p % B`` ("What is paged
    attention?", section "How it works").
  An append of ``n`` tokens is all-or-nothing: if the pool cannot supply every
  block it needs, nothing changes and ``OutOfBlocks`` is raised.
* ``free`` returns every block of the sequence's table, decrementing in reverse
  table order (the order is open on the pages; reverse order makes the worked
  example's request C receive P0 then P1, as the example states).
* Preemption by swapping ("PagedAttention — how vLLM stopped wasting 80%...",
  section "Preemption: what happens when memory runs out anyway": copy the
  preempted sequence's blocks out to CPU RAM, and back into freshly allocated
  GPU blocks when it resumes; "PagedAttention and vLLM: Virtual Memory for the
  KV Cache", section "L3": preemption is all-or-nothing per sequence):
  ``swap_out`` returns the sequence's table (the blocks whose contents go to
  host memory, in logical order) and gives every block back as ``free`` does,
  keeping the sequence's length; ``swap_in`` gives it ``ceil(length / B)``
  newly allocated blocks, all or nothing, in logical order.  A swapped-out
  sequence cannot be appended to, forked or exported until it is swapped in.

Sequence ids are handed out 0, 1, 2, ... and never reused.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple


class OutOfBlocks(RuntimeError):
    pass


class InvalidOperation(ValueError):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int,
                 pop_order: Optional[Sequence[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise InvalidOperation("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if pop_order is None else [int(x) for x in pop_order]
        if sorted(order) != list(range(num_blocks)):
            raise InvalidOperation("pop_order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self._free: List[int] = order[::-1]          # top of the stack is the end
        self.refcount: List[int] = [0] * num_blocks
        self.tables: dict = {}
        self.lengths: dict = {}
        self.swapped: set = set()
        self._next_seq = 0

    # --- free list and refcounts -------------------------------------------------
    def num_free(self) -> int:
        return len(self._free)

    def alloc(self) -> int:
        if not self._free:
            raise OutOfBlocks("no free block")
        b = self._free.pop()
        self.refcount[b] = 1
        return b

    def incref(self, b: int) -> None:
        if not (0 <= b < self.num_blocks) or self.refcount[b] <= 0:
            raise InvalidOperation(f"incref of unallocated block {b}")
        self.refcount[b] += 1

    def decref(self, b: int) -> None:
        if not (0 <= b < self.num_blocks) or self.refcount[b] <= 0:
            raise InvalidOperation(f"decref of unallocated block {b}")
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self._free.append(b)

    # --- sequences ---------------------------------------------------------------
    def create(self) -> int:
        sid = self._next_seq
        self._next_seq += 1
        self.tables[sid] = []
        self.lengths[sid] = 0
        return sid

    def fork(self, parent: int) -> int:
        self._check_resident(parent)
        child = self.create()
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for b in self.tables[child]:
            self.incref(b)
        return child

    def free(self, sid: int) -> None:
        self._check_seq(sid)
        for b in reversed(self.tables[sid]):
            self.decref(b)
        del self.tables[sid]
        del self.lengths[sid]
        self.swapped.discard(sid)

    def swap_out(self, sid: int) -> List[int]:
        """Preempt ``sid``: its table (blocks to copy to host, logical order); every
        block is given back (reverse order); the length is kept."""
        self._check_resident(sid)
        table = list(self.tables[sid])
        for b in reversed(table):
            self.decref(b)
        self.tables[sid] = []
        self.swapped.add(sid)
        return table

    def swap_in(self, sid: int) -> List[int]:
        """Resume ``sid``: ``ceil(length / B)`` fresh blocks (all or nothing)."""
        self._check_seq(sid)
        if sid not in self.swapped:
            raise InvalidOperation(f"sequence {sid} is not swapped out")
        n = -(-self.lengths[sid] // self.block_size)
        if n > self.num_free():
            raise OutOfBlocks("pool cannot hold the swapped-in sequence")
        table = [self.alloc() for _ in range(n)]
        self.tables[sid] = table
        self.swapped.discard(sid)
        return table

    def blocks_needed(self, sid: int, n: int) -> int:
        """Blocks an append of ``n`` tokens would take from the free list."""
        self._check_resident(sid)
        B = self.block_size
        t = self.lengths[sid]
        table = self.tables[sid]
        need = 0
        for p in range(t, t + n):
            if p % B == 0:
                need += 1
            elif p == t and self.refcount[table[-1]] > 1:
                need += 1
        return need

    def append(self, sid: int, n: int) -> Tuple[List[int], List[Tuple[int, int]]]:
        """Append ``n`` tokens; returns (slots, copy-on-write (src, dst) pairs)."""
        self._check_seq(sid)
        if n < 0:
            raise InvalidOperation("negative token count")
        if self.blocks_needed(sid, n) > self.num_free():
            raise OutOfBlocks("pool cannot hold the appended tokens")
        B = self.block_size
        table = self.tables[sid]
        slots: List[int] = []
        cows: List[Tuple[int, int]] = []
        for _ in range(n):
            p = self.lengths[sid]
            if p % B == 0:
                table.append(self.alloc())
            elif self.refcount[table[-1]] > 1:
                old = table[-1]
                new = self.alloc()
                cows.append((old, new))
                self.decref(old)
                table[-1] = new
            slots.append(table[p // B] * B + p % B)
            self.lengths[sid] = p + 1
        return slots, cows

    def export_tables(self, seqs: Sequence[int], max_blocks: int):
        """Row-padded ``[len(seqs), max_blocks]`` table (padding 0) and context lengths."""
        import numpy as np
        tab = np.zeros((len(seqs), max_blocks), dtype=np.int32)
        ctx = np.zeros(len(seqs), dtype=np.int32)
        for r, sid in enumerate(seqs):
            self._check_resident(sid)
            t = self.tables[sid]
            if len(t) > max_blocks:
                raise InvalidOperation("table longer than max_blocks")
            tab[r, :len(t)] = t
            ctx[r] = self.lengths[sid]
        return tab, ctx

    def _check_seq(self, sid: int) -> None:
        if sid not in self.tables:
            raise InvalidOperation(f"unknown sequence {sid}")

    def _check_resident(self, sid: int) -> None:
        self._check_seq(sid)
        if sid in self.swapped:
            raise InvalidOperation(f"sequence {sid} is swapped out")

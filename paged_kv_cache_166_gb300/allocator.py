"""Python handle on the library's host block manager (pkv_allocator_* in the C ABI)."""
from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

import numpy as np

from . import _native as N

_I32P = ctypes.POINTER(ctypes.c_int32)


def _ptr(a: np.ndarray):
    # an int32 element passed for a POINTER(c_int32) argument is taken by reference,
    # which ctypes does faster than building a pointer object
    if a.nbytes == 0:
        return None
    if a.flags.writeable and a.flags.c_contiguous:
        return ctypes.c_int32.from_buffer(a)
    return a.ctypes.data_as(_I32P)


class BlockAllocator:
    """Free list, refcounts, fork, append with copy-on-write and free over a fixed pool.

    ``pop_order`` fixes which ids the free list hands out first (a permutation of
    ``range(num_blocks)``; ascending when omitted).
    """

    def __init__(self, num_blocks: int, block_size: int,
                 pop_order: Optional[Sequence[int]] = None):
        self._lib = N.lib()
        h = ctypes.c_void_p()
        order = None
        if pop_order is not None:
            order = np.ascontiguousarray(np.asarray(pop_order, dtype=np.int32))
            if order.shape != (num_blocks,):
                raise ValueError("pop_order must have num_blocks entries")
        N.check(self._lib.pkv_allocator_create(num_blocks, block_size,
                                               _ptr(order) if order is not None else None,
                                               ctypes.byref(h)))
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.pkv_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _out(self, fn, *args) -> int:
        v = ctypes.c_int32(0)
        N.check(fn(self._h, *args, ctypes.byref(v)))
        return v.value

    # blocks
    def alloc(self) -> int:
        return self._out(self._lib.pkv_block_alloc)

    def incref(self, b: int) -> None:
        N.check(self._lib.pkv_block_incref(self._h, b))

    def decref(self, b: int) -> None:
        N.check(self._lib.pkv_block_decref(self._h, b))

    def refcount(self, b: int) -> int:
        return self._out(self._lib.pkv_block_refcount, b)

    def num_free(self) -> int:
        return self._out(self._lib.pkv_num_free_blocks)

    # sequences
    def create(self) -> int:
        return self._out(self._lib.pkv_seq_create)

    def fork(self, parent: int) -> int:
        return self._out(self._lib.pkv_seq_fork, parent)

    def free(self, seq: int) -> None:
        N.check(self._lib.pkv_seq_free(self._h, seq))

    def blocks_needed(self, seq: int, n: int) -> int:
        return self._out(self._lib.pkv_seq_blocks_needed, seq, n)

    def append(self, seq: int, n: int) -> Tuple[np.ndarray, List[Tuple[int, int]]]:
        """Append n tokens; returns (slots int32 [n], [(src, dst)] copy-on-write pairs)."""
        slots = np.empty(max(n, 1), dtype=np.int32)
        pair = np.zeros(2, dtype=np.int32)
        ncow = ctypes.c_int32(0)
        N.check(self._lib.pkv_seq_append(self._h, seq, n, _ptr(slots), _ptr(pair),
                                         ctypes.byref(ncow)))
        cows = [(int(pair[0]), int(pair[1]))] if ncow.value else []
        return slots[:n], cows

    def append_one_each(self, seqs: Sequence[int]) -> Tuple[np.ndarray, List[Tuple[int, int]]]:
        """One decode step: one new position for each listed sequence (distinct ids),
        in list order, as append(seq, 1) for each would do, in one library call.
        Returns (slots int32 [k], [(src, dst)] copy-on-write pairs in list order);
        all or nothing."""
        ids = np.ascontiguousarray(seqs, dtype=np.int32)
        k = len(ids)
        slots = np.empty(max(k, 1), dtype=np.int32)
        pairs = np.empty(max(2 * k, 2), dtype=np.int32)
        ncow = ctypes.c_int32(0)
        N.check(self._lib.pkv_seq_append_one_each(self._h, _ptr(ids), k, _ptr(slots),
                                                  _ptr(pairs), ctypes.byref(ncow)))
        cows = [(int(pairs[2 * i]), int(pairs[2 * i + 1])) for i in range(ncow.value)]
        return slots[:k], cows

    def swap_out(self, seq: int) -> List[int]:
        """Preempt by swapping: the sequence's block ids (logical order), all given
        back to the pool; copy their contents out (paged_swap_out) before reuse."""
        buf = np.empty(max(len(self.table(seq)), 1), dtype=np.int32)
        n = ctypes.c_int32(0)
        N.check(self._lib.pkv_seq_swap_out(self._h, seq, _ptr(buf), len(buf), ctypes.byref(n)))
        return buf[:n.value].tolist()

    def swap_in(self, seq: int) -> List[int]:
        """Resume a swapped-out sequence: its fresh block ids (logical order)."""
        B = self.block_size
        buf = np.empty(max(-(-self.length(seq) // B), 1), dtype=np.int32)
        n = ctypes.c_int32(0)
        N.check(self._lib.pkv_seq_swap_in(self._h, seq, _ptr(buf), len(buf), ctypes.byref(n)))
        return buf[:n.value].tolist()

    def length(self, seq: int) -> int:
        return self._out(self._lib.pkv_seq_len, seq)

    def table(self, seq: int) -> List[int]:
        n = ctypes.c_int32(0)
        N.check(self._lib.pkv_seq_table(self._h, seq, None, 0, ctypes.byref(n)))
        buf = np.empty(max(n.value, 1), dtype=np.int32)
        N.check(self._lib.pkv_seq_table(self._h, seq, _ptr(buf), n.value, ctypes.byref(n)))
        return buf[:n.value].tolist()

    def export_tables(self, seqs: Sequence[int], max_blocks: int,
                      tables_out: Optional[np.ndarray] = None,
                      ctx_out: Optional[np.ndarray] = None):
        """Row-padded int32 [len(seqs), max_blocks] table (padding 0) and int32 lengths,
        written into ``tables_out`` / ``ctx_out`` when given (C-contiguous int32 arrays
        of those shapes, e.g. views of page-locked staging buffers)."""
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        tab = np.zeros((len(s), max_blocks), dtype=np.int32) if tables_out is None else tables_out
        ctx = np.zeros(len(s), dtype=np.int32) if ctx_out is None else ctx_out
        for a, shape in ((tab, (len(s), max_blocks)), (ctx, (len(s),))):
            if a.dtype != np.int32 or a.shape != shape or not a.flags.c_contiguous:
                raise ValueError(f"output must be C-contiguous int32 of shape {shape}")
        N.check(self._lib.pkv_export_tables(self._h, _ptr(s), len(s), max_blocks, _ptr(tab),
                                            _ptr(ctx)))
        return tab, ctx


class DecodeStepTables:
    """The host side of one decode step for a fixed set of sequences, every buffer
    and C argument bound once: one new position for each sequence
    (pkv_seq_append_one_each), then their tables and lengths exported
    (pkv_export_tables) into ``tables_out`` [k, max_blocks] and ``ctx_out`` [k]
    (C-contiguous int32 arrays, e.g. views of page-locked staging memory that the
    step then copies to the device).  Calling it costs two library calls and no
    allocation; it returns the step's slots (int32 [k], overwritten by the next
    call) and its copy-on-write pairs."""

    def __init__(self, alloc: BlockAllocator, seqs: Sequence[int], max_blocks: int,
                 tables_out: np.ndarray, ctx_out: np.ndarray):
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        k = len(ids)
        for a, shape in ((tables_out, (k, max_blocks)), (ctx_out, (k,))):
            if a.dtype != np.int32 or a.shape != shape or not a.flags.c_contiguous:
                raise ValueError(f"output must be C-contiguous int32 of shape {shape}")
        self.alloc = alloc  # keeps the block manager alive
        self._ids, self.slots = ids, np.empty(max(k, 1), dtype=np.int32)
        self._pairs = np.empty(max(2 * k, 2), dtype=np.int32)
        self._ncow = ctypes.c_int32(0)
        self._tab, self._ctx = tables_out, ctx_out
        lib = alloc._lib
        self._append = lib.pkv_seq_append_one_each
        self._export = lib.pkv_export_tables
        self._a_args = (alloc._h, _ptr(ids), k, _ptr(self.slots), _ptr(self._pairs),
                        ctypes.byref(self._ncow))
        self._e_args = (alloc._h, _ptr(ids), k, max_blocks, _ptr(tables_out), _ptr(ctx_out))
        self._k = k

    def __call__(self) -> Tuple[np.ndarray, List[Tuple[int, int]]]:
        rc = self._append(*self._a_args)
        if rc:
            N.check(rc)
        rc = self._export(*self._e_args)
        if rc:
            N.check(rc)
        n = self._ncow.value
        cows = [(int(self._pairs[2 * i]), int(self._pairs[2 * i + 1])) for i in range(n)] if n else []
        return self.slots[:self._k], cows


"""Pins of the oracle's preemption by swapping (block manager and block copies).

"Swapping — copy the preempted sequence's KV cache blocks out to CPU RAM, and
copy them back into freshly allocated GPU blocks when the sequence resumes"
("PagedAttention — how vLLM stopped wasting 80% of your GPU memory", section
"Preemption: what happens when memory runs out anyway"); "preemption is
all-or-nothing per sequence" ("PagedAttention and vLLM: Virtual Memory for the
KV Cache", section "L3").

* A sequence swapped out, its blocks reused and overwritten by others, then
  swapped back in reads exactly what it read before — gathered rows and fp64
  attention output bit-equal — through different physical ids.
* Refcounts and the pool stay consistent with sharing: a forked sibling keeps
  the shared blocks; only exclusive blocks return to the free list; free plus
  in-use always equals the pool.
* Swap-in is all-or-nothing; swapped-out sequences refuse append, fork and
  export; an immediate swap-out / swap-in pair restores the same table (the
  free list is a stack and blocks are released in reverse table order).
"""
import numpy as np
import pytest

from oracle import cache_ops, paged_attention as pa
from oracle.block_manager import BlockManager, InvalidOperation, OutOfBlocks


def _pool(NB, Hkv=2, B=4, D=8, seed=0):
    r = np.random.default_rng(seed)
    return r.standard_normal((NB, Hkv, B, D)), r.standard_normal((NB, Hkv, B, D))


def _write(mgr, kc, vc, sid, n, r):
    slots, cows = mgr.append(sid, n)
    if cows:
        cache_ops.copy_blocks(kc, vc, np.asarray(cows))
    Hkv, D = kc.shape[1], kc.shape[3]
    cache_ops.kv_write(r.standard_normal((n, Hkv, D)), r.standard_normal((n, Hkv, D)),
                       slots, kc, vc)


def _in_use(mgr):
    return sum(1 for c in mgr.refcount if c > 0)


def test_round_trip_through_host_with_reuse_in_between():
    B, NB = 4, 40
    r = np.random.default_rng(1)
    kc, vc = _pool(NB, B=B)
    mgr = BlockManager(NB, B, r.permutation(NB))
    a = mgr.create()
    _write(mgr, kc, vc, a, 13, r)
    b = mgr.fork(a)                       # shares a's 4 blocks
    _write(mgr, kc, vc, b, 6, r)          # copy-on-write of the partial block, then more
    c = mgr.create()
    _write(mgr, kc, vc, c, 9, r)
    t = mgr.lengths[b]
    before_rows = [pa.gather_sequence(kc, mgr.tables[b], t, g) for g in range(2)]
    q = r.standard_normal((1, 4, 8))
    tab, ctx = mgr.export_tables([b], 8)
    before_out = pa.paged_attention(q, kc, vc, tab, ctx, 0.3)

    ids = mgr.swap_out(b)
    host_k, host_v = cache_ops.swap_out_blocks(kc, vc, ids)
    assert mgr.tables[b] == [] and mgr.lengths[b] == t
    # others take the released blocks and overwrite them
    d = mgr.create()
    _write(mgr, kc, vc, d, 4 * mgr.num_free() - 1, r)
    mgr.free(d)
    new_ids = mgr.swap_in(b)
    cache_ops.swap_in_blocks(host_k, host_v, new_ids, kc, vc)
    assert len(new_ids) == len(ids) and new_ids != ids

    after_rows = [pa.gather_sequence(kc, mgr.tables[b], t, g) for g in range(2)]
    for x, y in zip(before_rows, after_rows):
        assert np.array_equal(x, y)
    tab, ctx = mgr.export_tables([b], 8)
    assert np.array_equal(pa.paged_attention(q, kc, vc, tab, ctx, 0.3), before_out)
    # the sequence is an ordinary resident one again
    _write(mgr, kc, vc, b, 3, r)
    assert mgr.lengths[b] == t + 3


def test_refcounts_with_sharing():
    B, NB = 4, 20
    mgr = BlockManager(NB, B)
    a = mgr.create()
    mgr.append(a, 8)                      # two full blocks
    b = mgr.fork(a)                       # both blocks shared
    mgr.append(b, 5)                      # b: two private blocks more
    shared = list(mgr.tables[a])
    private = mgr.tables[b][2:]
    free0 = mgr.num_free()
    ids = mgr.swap_out(b)
    assert ids == shared + private
    assert all(mgr.refcount[x] == 1 for x in shared)     # still held by a
    assert all(mgr.refcount[x] == 0 for x in private)
    assert mgr.num_free() == free0 + len(private)
    assert mgr.num_free() + _in_use(mgr) == NB
    new = mgr.swap_in(b)
    assert len(new) == 4 and all(mgr.refcount[x] == 1 for x in new)
    assert not set(new) & set(shared)                      # private copies now
    assert mgr.num_free() + _in_use(mgr) == NB


def test_swap_in_is_all_or_nothing():
    B, NB = 4, 6
    mgr = BlockManager(NB, B)
    a = mgr.create()
    mgr.append(a, 16)
    mgr.swap_out(a)
    b = mgr.create()
    mgr.append(b, 12)                     # leaves 3 free, a needs 4
    free0, tables0 = mgr.num_free(), dict(mgr.tables)
    with pytest.raises(OutOfBlocks):
        mgr.swap_in(a)
    assert mgr.num_free() == free0 and mgr.tables == tables0 and a in mgr.swapped
    mgr.free(b)
    assert len(mgr.swap_in(a)) == 4


def test_swapped_sequence_refuses_resident_operations():
    mgr = BlockManager(8, 4)
    a = mgr.create()
    mgr.append(a, 5)
    mgr.swap_out(a)
    for op in (lambda: mgr.append(a, 1), lambda: mgr.fork(a), lambda: mgr.export_tables([a], 4),
               lambda: mgr.swap_out(a), lambda: mgr.blocks_needed(a, 1)):
        with pytest.raises(InvalidOperation):
            op()
    mgr.free(a)                            # a swapped sequence can be dropped
    assert mgr.num_free() == 8
    b = mgr.create()
    with pytest.raises(InvalidOperation):
        mgr.swap_in(b)                     # not swapped out


def test_immediate_round_trip_restores_the_table():
    mgr = BlockManager(30, 4, np.random.default_rng(4).permutation(30))
    a = mgr.create()
    mgr.append(a, 23)
    table = list(mgr.tables[a])
    assert mgr.swap_out(a) == table
    assert mgr.swap_in(a) == table


def test_empty_sequence_swaps_nothing():
    mgr = BlockManager(4, 4)
    a = mgr.create()
    assert mgr.swap_out(a) == [] and mgr.swap_in(a) == []

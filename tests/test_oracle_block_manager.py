"""Pins of the block-manager oracle: the pages' worked examples and closed forms.

* The three-request walk-through with block size 4 ("PagedAttention — how vLLM
  stopped wasting 80%...", section "A small worked example").
* The eight-request table, pool capacity and free count of "PagedAttention and
  vLLM: Virtual Memory for the KV Cache", "Scheme B".
* The parallel-sampling count of the same page ("A second calculation").
* Closed forms on random operation sequences: a sequence of t tokens holds
  ceil(t/B) blocks ("What is paged attention?", "How it works"), wastes at most
  B-1 slots, refcounts add up to the table entries that point at each block,
  free + in-use = pool size, and appends that cannot be served change nothing.
"""
import numpy as np
import pytest

from oracle.block_manager import BlockManager, OutOfBlocks, InvalidOperation
from oracle import kv_bytes


def run_script(rows, make_manager):
    cfg = {}
    mgr = None
    names = {}
    last_cow = {}
    for row in rows:
        op, args = row[0], row[1:]
        if op in ("block_size", "num_blocks"):
            cfg[op] = int(args[0])
            continue
        if mgr is None:
            mgr = make_manager(cfg["num_blocks"], cfg["block_size"])
        if op == "create":
            names[args[0]] = mgr.create()
        elif op == "append":
            _, cows = mgr.append(names[args[0]], int(args[1]))
            last_cow[args[0]] = cows
        elif op == "fork":
            names[args[0]] = mgr.fork(names[args[1]])
        elif op == "free":
            mgr.free(names[args[0]])
        elif op == "table":
            assert list(mgr.tables[names[args[0]]]) == [int(x) for x in args[1:]], row
        elif op == "refcount":
            assert mgr.refcount[int(args[0])] == int(args[1]), row
        elif op == "free_count":
            assert mgr.num_free() == int(args[0]), row
        elif op == "cow":
            assert args[1] == "none" and last_cow[args[0]] == [], row
        else:
            raise AssertionError(row)
    return mgr


def test_worked_example_three_requests(golden):
    run_script(golden("worked_example_b4.txt"), BlockManager)


def test_constructed_scenario_eight_requests(golden):
    rows = golden("constructed_scenario_b16.txt")
    kv = {r[0]: r[1:] for r in rows if r[0] != "request"}
    reqs = [tuple(map(int, r[1:])) for r in rows if r[0] == "request"]
    B = int(kv["block_size"][0])
    pool = int(kv["pool_blocks"][0])
    # capacity: 24 GB / (16 tokens x 512 KB) blocks, x16 tokens
    assert B * int(kv["bytes_per_token_kb"][0]) == int(kv["block_kb"][0])
    assert 24 * 1024 * 1024 // int(kv["block_kb"][0]) == pool
    assert pool * B == int(kv["pool_tokens"][0])
    mgr = BlockManager(pool, B)
    tot_blocks = tot_slots = tot_tok = tot_waste = 0
    for length, blocks, slots, wasted in reqs:
        sid = mgr.create()
        got_slots, cows = mgr.append(sid, length)
        assert cows == []
        assert len(mgr.tables[sid]) == blocks == kv_bytes.blocks_for(length, B)
        assert blocks * B == slots
        assert kv_bytes.waste_slots(length, B) == wasted
        assert len(set(got_slots)) == length
        tot_blocks += blocks; tot_slots += slots; tot_tok += length; tot_waste += wasted
    assert tot_blocks == int(kv["total_blocks"][0])
    assert tot_slots == int(kv["total_slots"][0])
    assert tot_tok == int(kv["total_tokens"][0])
    assert tot_waste == int(kv["total_wasted"][0])
    assert round(100 * tot_waste / tot_slots, 1) == float(kv["wasted_percent"][0])
    assert mgr.num_free() == int(kv["free_after"][0])
    extra = int(kv["extra_request_blocks"][0])
    assert kv_bytes.blocks_for(int(kv["extra_request_len"][0]), B) == extra
    assert mgr.num_free() // extra == int(kv["extra_requests"][0])
    # Scheme A (contiguous reservation of max_len per request), same traffic
    max_len = int(kv["max_len"][0])
    reserved = 8 * max_len
    assert round(100 * (reserved - tot_tok) / reserved, 1) == float(kv["contiguous_waste_percent"][0])
    per_req_gb = max_len * 512 / 1e6
    assert int(24 / round(per_req_gb, 2)) == int(kv["contiguous_max_requests"][0])


def test_parallel_sampling_block_count(golden):
    kv = {r[0]: r[1:] for r in golden("parallel_sampling_b16.txt")}
    B = int(kv["block_size"][0]); P = int(kv["prompt_len"][0])
    n = int(kv["samples"][0]); c = int(kv["completion_len"][0])
    assert n * (P + c) == int(kv["unshared_tokens"][0])
    assert kv_bytes.blocks_for(P, B) == int(kv["prompt_blocks"][0])
    assert kv_bytes.blocks_for(c, B) == int(kv["completion_blocks_each"][0])
    mgr = BlockManager(1000, B)
    parent = mgr.create()
    mgr.append(parent, P)
    assert len(mgr.tables[parent]) == int(kv["prompt_blocks"][0])
    sids = [parent] + [mgr.fork(parent) for _ in range(n - 1)]
    assert all(mgr.refcount[b] == n for b in mgr.tables[parent])
    copies = 0
    for sid in sids:
        _, cows = mgr.append(sid, c)
        copies += len(cows)
    in_use = mgr.num_blocks - mgr.num_free()
    # exact count under these rules: 62 full prompt blocks + the partial block and its
    # n-1 copies + 12 further blocks per sample = 114, within the page's "~119"
    assert copies == n - 1 <= int(kv["max_copied_blocks"][0])
    assert in_use == (P // B) + n + n * ((c - (B - P % B)) // B + ((c - (B - P % B)) % B > 0))
    assert in_use == 114 <= int(kv["approx_total_blocks"][0])
    assert int(kv["approx_total_blocks"][0]) * B == int(kv["approx_total_slots"][0])
    unshared_blocks = n * kv_bytes.blocks_for(P + c, B)
    saving = 100 * (1 - int(kv["approx_total_slots"][0]) / int(kv["unshared_tokens"][0]))
    assert abs(saving - int(kv["saving_percent"][0])) < 1.0
    assert in_use < unshared_blocks
    # the prompt blocks still shared by all samples are never copied
    shared = set(mgr.tables[sids[0]][:P // B])
    for sid in sids[1:]:
        assert set(mgr.tables[sid][:P // B]) == shared


def _check_invariants(mgr):
    B = mgr.block_size
    counts = np.zeros(mgr.num_blocks, dtype=np.int64)
    for sid, table in mgr.tables.items():
        t = mgr.lengths[sid]
        assert len(table) == kv_bytes.blocks_for(t, B)
        assert 0 <= len(table) * B - t <= B - 1
        for b in table:
            counts[b] += 1
    assert list(counts) == list(mgr.refcount)
    in_use = int(np.sum(counts > 0))
    assert in_use + mgr.num_free() == mgr.num_blocks
    assert len(set(mgr._free)) == mgr.num_free()
    assert all(mgr.refcount[b] == 0 for b in mgr._free)


@pytest.mark.parametrize("seed", range(6))
def test_random_operation_sequences_keep_invariants(seed):
    r = np.random.default_rng(100 + seed)
    B = int(r.choice([1, 4, 16]))
    NB = int(r.integers(20, 80))
    mgr = BlockManager(NB, B, pop_order=r.permutation(NB))
    live = []
    for _ in range(400):
        op = r.integers(0, 10)
        if op < 2 or not live:
            live.append(mgr.create())
        elif op < 7:
            sid = live[r.integers(len(live))]
            n = int(r.integers(0, 2 * B + 3))
            before = (list(mgr.refcount), {k: list(v) for k, v in mgr.tables.items()},
                      dict(mgr.lengths), list(mgr._free))
            t0 = mgr.lengths[sid]
            try:
                slots, cows = mgr.append(sid, n)
            except OutOfBlocks:
                after = (list(mgr.refcount), {k: list(v) for k, v in mgr.tables.items()},
                         dict(mgr.lengths), list(mgr._free))
                assert after == before
                continue
            assert len(cows) <= 1
            table = mgr.tables[sid]
            for i, s in enumerate(slots):
                p = t0 + i
                assert s == table[p // B] * B + p % B
                assert mgr.refcount[table[p // B]] == 1 or p // B < len(table) - 1 or cows
        elif op < 8:
            live.append(mgr.fork(live[r.integers(len(live))]))
        else:
            sid = live.pop(r.integers(len(live)))
            mgr.free(sid)
        _check_invariants(mgr)


def test_written_blocks_are_private():
    # after an append returns, every slot it wrote sits in a block with refcount 1
    mgr = BlockManager(64, 4)
    a = mgr.create(); mgr.append(a, 6)
    kids = [mgr.fork(a) for _ in range(3)]
    for sid in [a] + kids:
        slots, _ = mgr.append(sid, 3)
        for s in slots:
            assert mgr.refcount[s // 4] == 1


def test_errors_leave_state_unchanged():
    mgr = BlockManager(3, 4)
    a = mgr.create()
    mgr.append(a, 9)           # 3 blocks
    with pytest.raises(OutOfBlocks):
        mgr.append(a, 4)
    assert mgr.lengths[a] == 9 and mgr.num_free() == 0
    with pytest.raises(InvalidOperation):
        mgr.decref(7)
    with pytest.raises(InvalidOperation):
        mgr.free(99)
    mgr.free(a)
    assert mgr.num_free() == 3
    with pytest.raises(InvalidOperation):
        mgr.decref(0)


def test_pop_order_is_honoured():
    order = [5, 2, 7, 0, 1, 3, 4, 6]
    mgr = BlockManager(8, 16, pop_order=order)
    got = [mgr.alloc() for _ in range(8)]
    assert got == order
    with pytest.raises(OutOfBlocks):
        mgr.alloc()

"""Pins of the cache-write / block-copy oracle and of the KV size arithmetic.

* Cache write: writing a sequence's tokens through the slots the block manager
  hands out, then reading the blocks of its table back in logical order
  (a reshape, not the slot formula), recovers the tokens exactly; slots not
  written keep their canary bits; padding slots (-1) write nothing.
* Block copy: a copy-on-write pair duplicates the whole block.
* KV sizes printed on the pages (tests/golden/kv_sizes.txt).
"""
import numpy as np

from oracle import cache_ops, kv_bytes
from oracle.block_manager import BlockManager


def test_write_then_read_back_in_logical_order():
    r = np.random.default_rng(0)
    B, Hkv, D, NB = 4, 3, 8, 20
    mgr = BlockManager(NB, B, pop_order=r.permutation(NB))
    kc = np.full((NB, Hkv, B, D), -7.25); vc = np.full((NB, Hkv, B, D), -7.25)
    seqs = {}
    for t in (5, 1, 12, 7):
        sid = mgr.create()
        k = r.standard_normal((t, Hkv, D)); v = r.standard_normal((t, Hkv, D))
        slots, cows = mgr.append(sid, t)
        assert cows == []
        cache_ops.kv_write(k, v, slots, kc, vc)
        seqs[sid] = (k, v)
    written = np.zeros((NB, B), dtype=bool)
    for sid, (k, v) in seqs.items():
        table = mgr.tables[sid]
        t = k.shape[0]
        back_k = kc[table].transpose(0, 2, 1, 3).reshape(-1, Hkv, D)[:t]
        back_v = vc[table].transpose(0, 2, 1, 3).reshape(-1, Hkv, D)[:t]
        assert np.array_equal(back_k, k) and np.array_equal(back_v, v)
        for j, b in enumerate(table):
            written[b, :min(B, t - j * B)] = True
    assert np.all(kc.transpose(0, 2, 1, 3)[~written] == -7.25)
    assert np.all(vc.transpose(0, 2, 1, 3)[~written] == -7.25)


def test_padding_slots_write_nothing():
    kc = np.zeros((2, 1, 4, 2)); vc = np.zeros((2, 1, 4, 2))
    k = np.ones((3, 1, 2)); v = 2 * np.ones((3, 1, 2))
    cache_ops.kv_write(k, v, [-1, 5, -1], kc, vc)
    assert kc.sum() == 2 and vc.sum() == 4
    assert np.all(kc[1, 0, 1] == 1) and np.all(vc[1, 0, 1] == 2)


def test_copy_on_write_duplicates_the_block():
    r = np.random.default_rng(1)
    kc = r.standard_normal((6, 2, 4, 3)); vc = r.standard_normal((6, 2, 4, 3))
    k0 = kc.copy(); v0 = vc.copy()
    cache_ops.copy_blocks(kc, vc, [[1, 4], [2, 5]])
    assert np.array_equal(kc[4], k0[1]) and np.array_equal(vc[5], v0[2])
    assert np.array_equal(kc[:4], k0[:4])


def test_printed_kv_sizes(golden):
    for row in golden("kv_sizes.txt"):
        kind, a = row[0], row[1:]
        if kind == "sequence":
            L, H, D, T, e, gb, tol = a
            got = kv_bytes.kv_cache_bytes(int(L), int(H), int(D), int(T), int(e)) / 1e9
            assert abs(got - float(gb)) <= float(tol)
            # "Double the sequence length, double the cache"
            assert kv_bytes.kv_cache_bytes(int(L), int(H), int(D), 2 * int(T), int(e)) == \
                2 * kv_bytes.kv_cache_bytes(int(L), int(H), int(D), int(T), int(e))
        elif kind == "batch":
            n, L, H, D, T, e, gb, _ = a
            got = int(n) * kv_bytes.kv_cache_bytes(int(L), int(H), int(D), int(T), int(e)) / 1e9
            assert got > float(gb)
        elif kind == "block_head_bytes":
            B, D, e, want = map(int, a)
            assert kv_bytes.kv_cache_bytes(1, 1, D, B, e) == want
        elif kind == "request_block":
            L, H, B, D, e, mb = map(int, a)
            got = kv_bytes.kv_cache_bytes(L, H, D, B, e) / 2 ** 20
            assert abs(got - mb) < 0.5
        elif kind == "per_token":
            L, hidden, e, kb = map(int, a)
            # hidden size = num_kv_heads x head_dim for the multi-head model of the scenario
            assert kv_bytes.kv_cache_bytes(L, 1, hidden, 1, e) == kb * 1024


def test_block_bounds():
    # "A request that has produced t tokens holds ceil(t/16) blocks ... at most 15 tokens"
    for t in range(1, 200):
        n = kv_bytes.blocks_for(t, 16)
        assert (n - 1) * 16 < t <= n * 16
        assert 0 <= kv_bytes.waste_slots(t, 16) <= 15
    # "A sequence at token 40 with block size 16 occupies three blocks"
    assert kv_bytes.blocks_for(40, 16) == 3
    # contiguous waste of a 200-token request against a 4,096-token maximum: 95%
    assert round(100 * (4096 - 200) / 4096) == 95

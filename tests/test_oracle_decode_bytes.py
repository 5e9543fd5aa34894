"""Pins of the oracle's decode byte model (``oracle.kv_bytes.decode_bytes``), the
algorithmic byte count that every decode GB/s figure divides by, and the check
that ``bench.attention_bytes`` (the bench's own count, which may not import the
oracle on its timed path) agrees with it.

The byte model is pinned against things other than its own formula:

* the KV size the pages print for one 13B-shaped request of 2,048 tokens
  ("PagedAttention — how vLLM stopped wasting 80% of your GPU memory", section
  "The KV cache": roughly 1.7 GB over 40 layers) and the ``ceil(t / 16)`` block
  count ("What is paged attention?", section "How it works");
* the elements the oracle's attention depends on, found by brute force: every
  cache row and every table entry is changed in turn and counted when the
  output changes, on small ragged batches (lengths ending inside a block, on a
  block boundary, two tokens), several block sizes and group sizes.  Lengths 0
  and 1 are left out of this count on purpose: with one token the output is its
  value row whatever its key (softmax of one score is 1), and with none the
  query is not needed, yet the byte model counts both, as the decode reads them;
* planted mistakes (padded block tails counted, the query/output rows dropped,
  the 16-bit query counted at the 8-bit cache's element size, one table entry
  per padded block of the longest sequence) each fail the brute-force count.
"""
import numpy as np
import pytest

import bench
from oracle import kv_bytes, paged_attention
from paged_kv_cache_166_gb300 import workloads as W


def _dependency_bytes(lens, Hq, Hkv, D, B, kv_elt, q_elt):
    """Bytes the oracle's attention depends on, found by brute force on one small
    batch: a cache row (one block, KV head and offset) counts when replacing it
    changes the output, a table entry counts when pointing it at a spare block
    changes the output; entries past the sequence's blocks hold an id outside the
    pool, which would raise if read.  Plus one length, and every query row read
    and output row written, per sequence."""
    r = np.random.default_rng(7)
    S = len(lens)
    nbs = [-(-int(t) // B) for t in lens]
    spare = 2
    NB = sum(nbs) + spare
    perm = r.permutation(NB)
    maxb = max(nbs) + 2
    tables = np.full((S, maxb), 10 ** 9, dtype=np.int64)    # outside the pool
    at = 0
    for s, n in enumerate(nbs):
        tables[s, :n] = perm[at:at + n]
        at += n
    spares = perm[at:]
    kc = r.standard_normal((NB, Hkv, B, D))
    vc = r.standard_normal((NB, Hkv, B, D))
    q = r.standard_normal((S, Hq, D))
    ctx = np.asarray(lens)

    def run(kc_, vc_, tables_):
        return paged_attention.paged_attention(q, kc_, vc_, tables_, ctx, 0.125)

    base = run(kc, vc, tables)
    rows = 0
    for cache in (kc, vc):
        for b in range(NB):
            for g in range(Hkv):
                for o in range(B):
                    keep = cache[b, g, o].copy()
                    cache[b, g, o] = 3.0 + r.standard_normal(D)
                    rows += int(not np.array_equal(run(kc, vc, tables), base))
                    cache[b, g, o] = keep
    entries = 0
    for s in range(S):
        for j in range(maxb):
            keep = tables[s, j]
            tables[s, j] = spares[0]
            try:
                changed = not np.array_equal(run(kc, vc, tables), base)
            finally:
                tables[s, j] = keep
            entries += int(changed)
    assert min(lens) >= 2
    return (rows * D * kv_elt + 4 * entries + 4 * S + 2 * S * Hq * D * q_elt), entries


CASES = [
    # lens, Hq, Hkv, D, B
    ([2, 17, 40, 16], 2, 2, 4, 16),
    ([5, 8, 9, 23], 8, 2, 4, 8),
    ([31, 32, 33, 2], 6, 2, 4, 32),
    ([3, 4, 7], 2, 1, 8, 4),
]


@pytest.mark.parametrize("lens,Hq,Hkv,D,B", CASES)
def test_bytes_equal_what_the_oracle_depends_on(lens, Hq, Hkv, D, B):
    for kv_elt, q_elt in ((2, 2), (4, 4), (1, 2)):
        got, entries = _dependency_bytes(lens, Hq, Hkv, D, B, kv_elt, q_elt)
        assert entries == sum(kv_bytes.blocks_for(t, B) for t in lens)
        want = kv_bytes.decode_bytes(lens, Hq, Hkv, D, kv_elt, B, q_elem_bytes=q_elt)
        assert want == got


def test_planted_mistakes_fail_the_brute_force_count():
    lens, Hq, Hkv, D, B = [2, 17, 40], 4, 2, 4, 16
    got, _ = _dependency_bytes(lens, Hq, Hkv, D, B, 1, 2)
    nb = [kv_bytes.blocks_for(t, B) for t in lens]
    padded = sum(2 * n * B * Hkv * D + 4 * n + 4 + 2 * Hq * D * 2 for n in nb)
    no_q_out = sum(2 * t * Hkv * D + 4 * n + 4 for t, n in zip(lens, nb))
    q_at_cache_elt = kv_bytes.decode_bytes(lens, Hq, Hkv, D, 1, B)
    tables_of_longest = sum(2 * t * Hkv * D + 4 * max(nb) + 4 + 2 * Hq * D * 2 for t in lens)
    for wrong in (padded, no_q_out, q_at_cache_elt, tables_of_longest):
        assert wrong != got


def test_one_13b_request_matches_the_printed_size():
    """One 2,048-token request of the 13B shape: its decode bytes per layer are the
    size formula for one layer (1/40 of the printed ~1.7 GB) plus 128 = 2048/16
    table entries, its length and one query and one output row per head."""
    t, L, H, D, e = 2048, 40, 40, 128, 2
    total = kv_bytes.decode_bytes([t], H, H, D, e, 16)
    kv = total - 4 * 128 - 4 - 2 * H * D * e
    assert kv == 2 * H * D * t * e == 41_943_040
    assert abs(L * kv / 1e9 - 1.7) < 0.05
    # block size only enters through the table entries
    assert kv_bytes.decode_bytes([t], H, H, D, e, 8) - total == 4 * (256 - 128)
    # no padded tail: 17 tokens cost one token more than 16, not a block more
    one = kv_bytes.decode_bytes([17], H, H, D, e, 16) - kv_bytes.decode_bytes([16], H, H, D, e, 16)
    assert one == 2 * H * D * e + 4


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
@pytest.mark.parametrize("block_size", [8, 16, 32])
def test_bench_byte_count_equals_the_oracle(name, block_size):
    w = W.WORKLOADS[name]
    lens = W.context_lengths(w)
    elt = {"f32": 4, "f16": 2, "bf16": 2}[w.dtype]
    args = (lens, w.num_q_heads, w.num_kv_heads, w.head_dim)
    assert bench.attention_bytes(*args, elt, block_size) == \
        kv_bytes.decode_bytes(*args, elt, block_size)
    if elt == 2:   # the 8-bit caches: one byte per K/V element, 16-bit q and out
        assert bench.attention_bytes(*args, 1, block_size, 2) == \
            kv_bytes.decode_bytes(*args, 1, block_size, q_elem_bytes=2)


def test_bench_byte_count_of_the_13b_batch():
    w = W.WORKLOADS["mha13b"]
    lens = W.context_lengths(w)
    assert int(lens.sum()) == 24_860
    assert kv_bytes.decode_bytes(lens, 40, 40, 128, 2, 16) == 510_450_108

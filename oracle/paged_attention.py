"""Single-token paged decode attention in fp64 — the oracle.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``): never imported by the library.

What is computed, for every sequence ``s`` and query head ``h``:

1. ``g = h // G`` with ``G = Hq / Hkv`` — query heads are grouped contiguously
   onto KV heads (the pages are silent on the GQA mapping; this is the plain
   reading: consecutive query heads share one KV head).
2. ``t = context_lens[s]`` — the number of cached tokens, the new token
   included (it is written before attention runs: "each decode step -> write the
   new token's K,V into the last block", "PagedAttention and vLLM: Virtual
   Memory for the KV Cache", section "L2 — Mechanism", allocation lifecycle).
3. for each position ``p < t``: ``slot(p) = block_table[p // B] * B + p % B``
   ("What is paged attention?", section "How it works"); the key and value of
   position ``p`` are ``K[slot // B, g, slot % B, :]`` and the same in V, the
   cache layout ``[num_blocks, num_kv_heads, block_size, head_dim]`` of
   "PagedAttention: How vLLM Borrowed Virtual Memory...", section "The Custom
   CUDA Kernel".
4. ``score_p = scale * q . k_p``;  ``w_p = exp(score_p - max score)``;
   ``out = sum_p w_p v_p / sum_p w_p`` — the softmax over all positions and the
   weighted sum of values, exactly the contiguous attention result ("PagedAttention
   — how vLLM stopped wasting 80%...", section "The PagedAttention kernel":
   "mathematically ... exactly the same attention"; FAQ "Does PagedAttention
   change the model's outputs?").

``t == 0`` has no definition on the pages; the oracle returns zeros for it.
All arithmetic is fp64; inputs of any float dtype are widened exactly.
"""
from __future__ import annotations

import numpy as np


def slot_of(block_table_row, p: int, block_size: int) -> int:
    """slot(p) = block_table[floor(p / B)] * B + (p mod B)."""
    return int(block_table_row[p // block_size]) * block_size + (p % block_size)


def gather_sequence(cache, block_table_row, t: int, kv_head: int) -> np.ndarray:
    """The ``[t, head_dim]`` fp64 rows of one sequence and KV head, read position by
    position through the block table."""
    cache = np.asarray(cache)
    B = cache.shape[2]
    p = np.arange(t)
    phys = np.asarray(block_table_row, dtype=np.int64)[p // B]
    off = p % B
    return np.asarray(cache[phys, kv_head, off, :], dtype=np.float64)


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale,
                    seqs=None) -> np.ndarray:
    """fp64 decode attention output ``[S, Hq, D]`` (rows of ``seqs`` only, others zero).

    q: ``[S, Hq, D]``; k_cache, v_cache: ``[NB, Hkv, B, D]``;
    block_tables: ``[S, max_blocks]`` physical ids; context_lens: ``[S]``;
    scale: the fp32 softmax scale, widened to fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    S, Hq, D = q.shape
    Hkv = np.asarray(k_cache).shape[1]
    G = Hq // Hkv
    sc = np.float64(np.float32(scale))
    out = np.zeros((S, Hq, D), dtype=np.float64)
    for s in (range(S) if seqs is None else seqs):
        t = int(context_lens[s])
        if t == 0:
            continue
        for g in range(Hkv):
            K = gather_sequence(k_cache, block_tables[s], t, g)
            V = gather_sequence(v_cache, block_tables[s], t, g)
            for h in range(g * G, (g + 1) * G):
                scores = sc * (K @ q[s, h])
                w = np.exp(scores - scores.max())
                out[s, h] = (w @ V) / w.sum()
    return out

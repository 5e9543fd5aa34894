"""Paged (chunked) prefill attention in fp64 — the oracle.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``): never imported by the library.

Prefill processes many prompt tokens of a sequence in one pass; chunked prefill
breaks a long prompt into chunks of a fixed token count interleaved with decode
steps, without changing how the KV cache is allocated ("PagedAttention: How
vLLM Borrowed Virtual Memory...", section "Walking Through the Lifecycle",
Prefill; section "RadixAttention ... Chunked prefill").  A paged KV cache is
what lets a chunk read the KV of the earlier chunks ("PagedAttention — how vLLM
stopped wasting 80%...", FAQ "Does this help the prompt-processing (prefill)
phase too?").

What is computed, the plain reading: sequence ``s`` has ``t = context_lens[s]``
tokens in the cache (its new chunk included, written before attention runs)
and a chunk of ``c = query_start[s+1] - query_start[s]`` queries, the last
``c`` positions: query row ``query_start[s] + i`` sits at position
``p = t - c + i`` and, for query head ``h`` of KV group ``g = h // G``, attends
causally to every position ``j <= p`` read through the block table:

    out[row, h] = sum_{j<=p} w_j V[slot(j), g] / sum_{j<=p} w_j,
    w_j = exp(scale * q[row, h] . K[slot(j), g] - max).

A whole-prompt prefill is the case ``c = t``.  All arithmetic is fp64.
"""
from __future__ import annotations

import numpy as np

from .paged_attention import gather_sequence


def paged_prefill_attention(q, k_cache, v_cache, block_tables, context_lens, query_start,
                            scale) -> np.ndarray:
    """fp64 output ``[T, Hq, D]`` for queries ``q [T, Hq, D]`` (T = query_start[-1])."""
    q = np.asarray(q, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = np.asarray(k_cache).shape[1]
    G = Hq // Hkv
    sc = np.float64(np.float32(scale))
    qs = np.asarray(query_start, dtype=np.int64)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    for s in range(len(qs) - 1):
        t = int(context_lens[s])
        c = int(qs[s + 1] - qs[s])
        if c == 0:
            continue
        for g in range(Hkv):
            K = gather_sequence(k_cache, block_tables[s], t, g)
            V = gather_sequence(v_cache, block_tables[s], t, g)
            for i in range(c):
                p = t - c + i
                for h in range(g * G, (g + 1) * G):
                    scores = sc * (K[:p + 1] @ q[qs[s] + i, h])
                    w = np.exp(scores - scores.max())
                    out[qs[s] + i, h] = (w @ V[:p + 1]) / w.sum()
    return out

"""Cache-write scatter and copy-on-write block copy — the oracle.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``): never imported by the library.

* ``kv_write``: for written token ``i`` with slot ``s = slot_mapping[i]``,
  ``K[s // B, h, s % B, :] = k[i, h, :]`` and the same for V, for every KV head
  ``h`` — a bit copy.  Each decode step writes the new token's K and V into its
  slot before attention reads the cache ("PagedAttention and vLLM: Virtual
  Memory for the KV Cache", section "L2 — Mechanism", allocation lifecycle;
  "PagedAttention: How vLLM Borrowed Virtual Memory...", section "Walking
  Through the Lifecycle", Decode).  A negative slot marks a padding token and
  is skipped (the pages are silent on padding; this is the library's
  convention).
* ``copy_blocks``: copy-on-write duplicates a whole physical block, K and V,
  from ``src`` to ``dst`` ("allocates a new physical block, copies the
  content", same page, section "Copy-on-Write for Beam Search and Parallel
  Sampling").
* ``swap_out_blocks`` / ``swap_in_blocks``: preemption by swapping copies a
  sequence's blocks out to host memory and back into freshly allocated blocks
  ("PagedAttention — how vLLM stopped wasting 80%...", section "Preemption:
  what happens when memory runs out anyway"): the host buffer holds the blocks
  in the order of the id list, each block whole (every KV head and slot).
"""
from __future__ import annotations

import numpy as np


def kv_write(k, v, slot_mapping, k_cache: np.ndarray, v_cache: np.ndarray) -> None:
    """Scatter ``k, v [T, Hkv, D]`` into ``k_cache, v_cache [NB, Hkv, B, D]`` in place."""
    B = k_cache.shape[2]
    for i, s in enumerate(np.asarray(slot_mapping).tolist()):
        if s < 0:
            continue
        k_cache[s // B, :, s % B, :] = k[i]
        v_cache[s // B, :, s % B, :] = v[i]


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, src_dst_pairs) -> None:
    """Copy block ``src`` onto block ``dst`` (all KV heads, all slots) for each pair, in order."""
    for src, dst in np.asarray(src_dst_pairs, dtype=np.int64).reshape(-1, 2).tolist():
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]


def swap_out_blocks(k_cache: np.ndarray, v_cache: np.ndarray, block_ids):
    """Host copies ``[n, ...]`` of the K and V blocks ``block_ids``, in that order."""
    ids = np.asarray(block_ids, dtype=np.int64)
    return k_cache[ids].copy(), v_cache[ids].copy()


def swap_in_blocks(host_k: np.ndarray, host_v: np.ndarray, block_ids, k_cache: np.ndarray,
                   v_cache: np.ndarray) -> None:
    """Block ``block_ids[i]`` of each cache becomes host block ``i``."""
    for i, b in enumerate(np.asarray(block_ids, dtype=np.int64).tolist()):
        k_cache[b] = host_k[i]
        v_cache[b] = host_v[i]

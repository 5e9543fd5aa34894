"""KV-cache size and block arithmetic — the oracle.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``): never imported by the library.

* KV bytes of one sequence: ``2 * num_layers * num_kv_heads * head_dim *
  seq_len * bytes_per_element`` — the leading 2 counts K and V
  ("PagedAttention and vLLM: Virtual Memory for the KV Cache", FAQ answer on
  whether paging reduces the cache a sequence needs).
* Blocks held by a sequence of ``t`` tokens: ``ceil(t / B)``, so at most one
  partially filled block ("What is paged attention?", section "How it works").
* Waste of a sequence: ``ceil(t / B) * B - t`` slots, at most ``B - 1``
  ("PagedAttention and vLLM...", property 1 "Internal fragmentation is bounded
  by one block").
* Decode-attention bytes read for one sequence, used as the algorithmic byte
  count of the measured metric: the K and V rows of the ``t`` cached tokens of
  every KV head (padded block tails are not counted), the ``ceil(t / B)``
  int32 table entries, the context length, and one query and one output row
  per query head.  With an 8-bit cache the K/V rows take one byte per element
  while the query and output rows keep their 16-bit type ("PagedAttention —
  how vLLM stopped wasting 80%...", FAQ "How does this relate to
  quantization?": the cache elements are what shrink), so the query/output
  element size is a separate argument that defaults to the cache's.
"""
from __future__ import annotations


def kv_cache_bytes(num_layers: int, num_kv_heads: int, head_dim: int, seq_len: int,
                   bytes_per_element: int) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * seq_len * bytes_per_element


def blocks_for(t: int, block_size: int) -> int:
    return -(-int(t) // int(block_size))


def waste_slots(t: int, block_size: int) -> int:
    return blocks_for(t, block_size) * block_size - int(t)


def decode_bytes(context_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 elem_bytes: int, block_size: int, q_elem_bytes: int | None = None) -> int:
    q_elem_bytes = elem_bytes if q_elem_bytes is None else q_elem_bytes
    total = 0
    for t in context_lens:
        t = int(t)
        total += 2 * t * num_kv_heads * head_dim * elem_bytes
        total += 4 * blocks_for(t, block_size) + 4
        total += 2 * num_q_heads * head_dim * q_elem_bytes
    return total

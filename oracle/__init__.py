"""fp64 CPU oracle of the paged KV-cache hot path: decode and prefill attention, the
cache writes (16-bit and 8-bit), block copies, swapping and the block manager.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference legs of ``bench.py`` may import or run anything in
this package.  The library (``paged_kv_cache_166_gb300``) never imports it and
shares no code with it; the two meet only in the seeded input generators of
``paged_kv_cache_166_gb300.workloads``, which hold none of the method's
arithmetic.

Each function is the plain definition of what the paged decode path computes,
written from the pages that describe PagedAttention:

* ``paged_attention``  — decode attention read through a block table
  ("PagedAttention — how vLLM stopped wasting 80% of your GPU memory",
  section "The PagedAttention kernel: computing attention over scattered
  blocks"; slot formula from "What is paged attention?", section "How it
  works").
* ``cache_ops``        — the cache-write scatter, the copy-on-write block copy and
  the block copies of swapping to and from host memory ("PagedAttention — how
  vLLM stopped wasting 80%...", section "Preemption: what happens when memory
  runs out anyway").
* ``block_manager``    — free list, refcounts, fork, append with copy-on-write,
  free ("PagedAttention: How vLLM Borrowed Virtual Memory...", sections
  "The OS-Inspired Insight" and "Walking Through the Lifecycle").
* ``kv_bytes``         — the KV-cache size formula and block arithmetic
  ("PagedAttention and vLLM: Virtual Memory for the KV Cache", summary FAQ).
* ``prefill``          — paged (chunked) prefill attention: a chunk of queries
  attending causally through the block table ("PagedAttention: How vLLM
  Borrowed Virtual Memory...", section "Walking Through the Lifecycle").
* ``fp8``              — the fp8 (E4M3) quantised KV cache: code table, the
  quantising cache write and attention over the dequantised values
  ("PagedAttention — how vLLM stopped wasting 80%...", FAQ "How does this
  relate to quantization?").
* ``int8``             — the int8 quantised KV cache (symmetric codes in
  [-127, 127], per-KV-head scales, the fp8 cache's layouts; same FAQ).

Every function here is pinned by ``tests/test_oracle_*.py`` against values the
pages print, library routines on special cases, closed forms and invariants.
"""

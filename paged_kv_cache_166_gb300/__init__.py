"""GB300-native paged KV-cache decode path (PagedAttention hot path).

Public API (all device work runs in libpkv.so's sm_103a kernels):

* ``paged_kv_write(k, v, slot_mapping, k_cache, v_cache)``
* ``paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, out)``
* ``paged_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out)``
  — the cache write of each sequence's new token, then the attention, from one call
* ``paged_copy_blocks(k_cache, v_cache, src_dst_pairs)``; ``paged_copy_blocks_layers(k_caches,
  v_caches, src_dst_pairs)`` — the same copies in every layer's caches, one launch
* ``paged_prefill_attention(q, k_cache, v_cache, block_tables, context_lens, query_start, scale, out)``
  — causal attention of each sequence's chunk of new prompt tokens
* fp8 (E4M3) cache with per-KV-head scales: ``paged_kv_write_fp8``,
  ``paged_decode_attention_fp8``, ``paged_decode_step_fp8``; the int8 cache:
  ``paged_kv_write_int8``, ``paged_decode_attention_int8``, ``paged_decode_step_int8``
* ``paged_swap_out`` / ``paged_swap_in`` — blocks to and from pinned host memory
  (preemption by swapping, with ``BlockAllocator.swap_out`` / ``swap_in``);
  ``paged_swap_out_layers`` / ``paged_swap_in_layers`` — every layer's caches, one launch
* ``BlockAllocator`` — host block manager (free list, refcounts, fork, CoW, free);
  ``DecodeStepTables`` — one decode step's appends and table export, pre-bound
* ``decode_status(workspace)`` — the device-side status bits of the decode kernels;
  ``wait_timeout_selftest()`` — the kernels' bounded wait made to run out on purpose

The library is loaded on first use; importing this package needs no GPU.
"""
from .allocator import BlockAllocator, DecodeStepTables  # noqa: F401
from ._native import OutOfBlocks, PkvError  # noqa: F401


def __getattr__(name):
    # torch-facing ops are imported lazily so that host-only users (the block
    # manager, the workload generators) do not need torch's CUDA runtime.
    if name in ("paged_kv_write", "paged_decode_attention", "paged_decode_step",
                "paged_copy_blocks", "paged_copy_blocks_layers", "paged_kv_write_fp8", "paged_decode_attention_fp8",
                "paged_decode_step_fp8", "paged_kv_write_int8", "paged_decode_attention_int8",
                "paged_decode_step_int8", "paged_swap_out", "paged_swap_in", "paged_swap_out_layers", "paged_swap_in_layers",
                "paged_prefill_attention",
                "decode_status", "workspace_bytes", "default_num_warps", "get_workspace",
                "wait_timeout_selftest"):
        from . import ops
        return getattr(ops, name)
    raise AttributeError(name)

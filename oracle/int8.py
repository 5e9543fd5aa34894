"""int8 KV-cache quantisation — the oracle.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``): never imported by the library.

The pages list int8 beside fp8 as the narrower element type of a quantised KV
cache, orthogonal to paging ("PagedAttention — how vLLM stopped wasting 80% of
your GPU memory", FAQ "How does this relate to quantization?").  They fix no
format.  The reading taken here is the plain symmetric one:

* a code is a signed 8-bit integer in [-127, 127] (two's complement; -128 is
  never written), and reads back as ``code * scale``;
* one fp32 scale per KV head for K and one for V, as for the fp8 cache;
* ``code = clamp(round(x / scale), -127, 127)`` with the quotient a correctly
  rounded fp32 division, rounded to the nearest integer with ties to the even
  one; infinities saturate, NaN gives code 0 (an integer code has no NaN).

Layouts are the fp8 cache's (block size 16): K ``[num_blocks, num_kv_heads, 16,
head_dim]``; V tiles transposed ``[num_blocks, num_kv_heads, head_dim, 16]``
with token ``t`` at byte ``V_POS[t]`` of each head_dim row.  Attention over the
int8 cache is the fp64 decode attention over the dequantised values.
"""
from __future__ import annotations

import numpy as np

from .fp8 import BLOCK, V_POS

MAX_CODE = 127


def quantize(x, scale) -> np.ndarray:
    """int8 codes of ``fp32(x) / fp32(scale)``: the fp32 quotient rounded to the
    nearest integer (ties to even), clamped to [-127, 127]; NaN -> 0."""
    q = np.asarray(x, dtype=np.float32) / np.asarray(scale, dtype=np.float32)
    q = q.astype(np.float64)
    r = np.rint(q)                      # IEEE round to nearest, ties to even
    r = np.clip(np.nan_to_num(r, nan=0.0, posinf=MAX_CODE, neginf=-MAX_CODE),
                -MAX_CODE, MAX_CODE)
    return r.astype(np.int8)


def decode(codes) -> np.ndarray:
    """int8 codes -> their values (before the scale) as fp64."""
    return np.asarray(codes).astype(np.int8).astype(np.float64)


def kv_write_int8(k, v, slot_mapping, k_scale, v_scale, k_cache: np.ndarray,
                  v_cache: np.ndarray) -> None:
    """Quantise and scatter ``k, v [T, Hkv, D]`` into the int8 caches in place:
    ``K8[s // 16, h, s % 16, :] = quantize(k[i, h, :], k_scale[h])`` and
    ``V8[s // 16, h, :, V_POS[s % 16]] = quantize(v[i, h, :], v_scale[h])``;
    negative slots are padding and skipped."""
    B = k_cache.shape[2]
    assert B == BLOCK and v_cache.shape[3] == BLOCK
    ks = np.asarray(k_scale, dtype=np.float32)[:, None]
    vs = np.asarray(v_scale, dtype=np.float32)[:, None]
    k32 = np.asarray(k, dtype=np.float32)
    v32 = np.asarray(v, dtype=np.float32)
    for i, s in enumerate(np.asarray(slot_mapping).tolist()):
        if s < 0:
            continue
        k_cache[s // B, :, s % B, :] = quantize(k32[i], ks)
        v_cache[s // B, :, :, V_POS[s % B]] = quantize(v32[i], vs)


def gather_int8(k_cache, v_cache, k_scale, v_scale, block_table_row, t: int, kv_head: int):
    """The fp64 ``[t, head_dim]`` K and V rows of one sequence and KV head, read
    position by position through the block table and dequantised."""
    B = k_cache.shape[2]
    p = np.arange(t)
    phys = np.asarray(block_table_row, dtype=np.int64)[p // B]
    off = p % B
    ks = np.float64(np.float32(k_scale[kv_head]))
    vs = np.float64(np.float32(v_scale[kv_head]))
    k = decode(np.asarray(k_cache)[phys, kv_head, off, :]) * ks
    v = decode(np.asarray(v_cache)[phys, kv_head, :, V_POS[off]]) * vs
    return k, v


def paged_attention_int8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                         scale: float, seqs=None) -> np.ndarray:
    """Decode attention over the int8 caches: the fp64 attention (as in
    ``paged_attention``) over their dequantised values; rows of ``seqs`` only."""
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
            K, V = gather_int8(k_cache, v_cache, k_scale, v_scale, block_tables[s], t, g)
            for h in range(g * G, (g + 1) * G):
                scores = sc * (K @ q[s, h])
                w = np.exp(scores - scores.max())
                out[s, h] = (w @ V) / w.sum()
    return out

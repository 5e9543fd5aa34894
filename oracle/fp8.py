"""fp8 (E4M3) KV-cache quantisation — the oracle.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``): never imported by the library.

The pages name a quantised KV cache — K and V stored in 8 bits instead of 16,
halving the bytes per element — as orthogonal to and composable with paging
("PagedAttention — how vLLM stopped wasting 80% of your GPU memory", FAQ "How
does this relate to quantization?"; "PagedAttention and vLLM: Virtual Memory
for the KV Cache", FAQ on the size formula: "KV-cache quantization to halve
bytes per element").  They fix no format.  The reading taken here:

* element format E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
  bits; exponent field 0 encodes subnormals ``m * 2^-9``; the all-ones pattern
  ``S.1111.111`` is NaN and there is no infinity, so the largest finite value
  is ``1.75 * 2^8 = 448``;
* one fp32 scale per KV head for K and one for V; a cache element holds
  ``code = E4M3(x / scale)`` — the quotient taken in fp32 (correctly rounded),
  then rounded to the nearest E4M3 value, ties to an even code, and saturated to
  +-448 beyond the range; NaN gives the code 0x7F;
* it reads back as ``decode(code) * scale``.

Layouts (block size 16): the K cache keeps ``[num_blocks, num_kv_heads, 16,
head_dim]``; the V cache stores each (block, KV head) tile transposed,
``[num_blocks, num_kv_heads, head_dim, 16]``, and inside each 16-byte head_dim
row token ``t`` sits at byte ``V_POS[t]`` — the order ``0 1 8 9 2 3 10 11 4 5
12 13 6 7 14 15`` (byte ``j`` holds token ``V_TOKEN[j]``), which a tensor-core
kernel reads in the token pairs of its score fragments.  Attention over the fp8
cache is the fp64 decode attention (the definition ``paged_attention`` follows)
over the dequantised values.
"""
from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0
NAN_CODE = 0x7F
BLOCK = 16
# byte j of a V head_dim row holds token V_TOKEN[j]; token t sits at byte V_POS[t]
V_TOKEN = np.array([0, 1, 8, 9, 2, 3, 10, 11, 4, 5, 12, 13, 6, 7, 14, 15])
V_POS = np.argsort(V_TOKEN)


def decode(codes) -> np.ndarray:
    """E4M3 codes (uint8) -> their exact values as fp64."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


_FINITE = decode(np.arange(0x7F))  # magnitudes of codes 0x00..0x7E, increasing


def encode(x) -> np.ndarray:
    """Values (taken as fp64; callers pass the fp32 quotient) -> E4M3 codes:
    round to nearest, ties to the even code, saturate beyond +-448, NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # the two neighbours of a among the finite magnitudes
    hi = np.clip(np.searchsorted(_FINITE, a, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo = np.abs(a - _FINITE[lo])
    d_hi = np.abs(_FINITE[hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo)
    mag = np.where(a >= MAX_FINITE, 0x7E, mag)
    code = np.where(np.signbit(x), mag | 0x80, mag)
    code = np.where(np.isnan(x), NAN_CODE, code)
    return code.astype(np.uint8)


def quantize(x, scale) -> np.ndarray:
    """code = E4M3(fp32(x) / fp32(scale)) with the division in fp32."""
    q = np.asarray(x, dtype=np.float32) / np.asarray(scale, dtype=np.float32)
    return encode(q.astype(np.float32))


def kv_write_fp8(k, v, slot_mapping, k_scale, v_scale, k_cache: np.ndarray,
                 v_cache: np.ndarray) -> None:
    """Quantise and scatter ``k, v [T, Hkv, D]`` into the fp8 caches in place:
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


def gather_fp8(k_cache, v_cache, k_scale, v_scale, block_table_row, t: int, kv_head: int):
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


def paged_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                        scale: float, seqs=None) -> np.ndarray:
    """Decode attention over the fp8 caches: the fp64 attention (as in
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
            K, V = gather_fp8(k_cache, v_cache, k_scale, v_scale, block_tables[s], t, g)
            for h in range(g * G, (g + 1) * G):
                scores = sc * (K @ q[s, h])
                w = np.exp(scores - scores.max())
                out[s, h] = (w @ V) / w.sum()
    return out

"""Seeded synthetic inputs for the paged decode workloads.

This module only draws random numbers and describes workload shapes.  It holds
none of the paged-attention arithmetic (no block counts, no slot formula, no
softmax): both the CUDA path and the fp64 oracle receive the same draws from
here and each applies its own arithmetic to them.

Workload shapes follow the five decode configurations the library is measured
on (tiny fp32 check, 13B-shaped MHA, 70B-shaped GQA, shared-prefix parallel
sampling, long-context GQA).  No public dataset is involved: the heavy-tailed
request lengths the pages describe ("PagedAttention: How vLLM Borrowed Virtual
Memory...", section "The Fragmentation Problem") are stood in for by
lognormal draws.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# Streams drawn from one workload seed.  Each stream gets its own generator so
# that drawing one tensor never shifts the values of another.
STREAM_LENGTHS = 0
STREAM_POOL_ORDER = 1
STREAM_Q = 2
STREAM_K_POOL = 3
STREAM_V_POOL = 4
STREAM_K_NEW = 5
STREAM_V_NEW = 6
STREAM_SUFFIX = 7
STREAM_SCALES = 8


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and draw recipe of one decode batch."""

    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str  # "f32" | "f16" | "bf16"
    block_size: int = 16
    num_seqs: int = 0
    # length recipe: "fixed" | "lognormal" | "uniform" | "prefix"
    length_kind: str = "fixed"
    fixed_lengths: tuple = ()
    median: float = 0.0
    sigma: float = 0.0
    lo: int = 1
    hi: int = 1
    # spare fraction of the physical pool beyond what the batch holds
    pool_spare: float = 0.10
    fixed_pool_blocks: int = 0
    # shared-prefix recipe
    num_prompts: int = 0
    samples_per_prompt: int = 0
    prompt_len: int = 0
    suffix_lo: int = 0
    suffix_hi: int = 0
    # number of new tokens written through the cache-write step per batch
    # (one per sequence for a decode step)
    writes_new_tokens: bool = True

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / np.sqrt(self.head_dim)))


WORKLOADS = {
    "tiny": Workload(
        name="tiny", seed=0, num_q_heads=4, num_kv_heads=4, head_dim=64, dtype="f32",
        num_seqs=4, length_kind="fixed", fixed_lengths=(1, 17, 40, 100),
        fixed_pool_blocks=32),
    "mha13b": Workload(
        name="mha13b", seed=1, num_q_heads=40, num_kv_heads=40, head_dim=128, dtype="f16",
        num_seqs=64, length_kind="lognormal", median=300.0, sigma=1.0, lo=1, hi=2048),
    "gqa70b": Workload(
        name="gqa70b", seed=2, num_q_heads=64, num_kv_heads=8, head_dim=128, dtype="bf16",
        num_seqs=256, length_kind="lognormal", median=1024.0, sigma=1.2, lo=1, hi=8192),
    "prefix": Workload(
        name="prefix", seed=3, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
        num_seqs=256, length_kind="prefix", num_prompts=32, samples_per_prompt=8,
        prompt_len=1000, suffix_lo=0, suffix_hi=512, writes_new_tokens=False),
    "longctx": Workload(
        name="longctx", seed=4, num_q_heads=64, num_kv_heads=8, head_dim=128, dtype="bf16",
        num_seqs=8, length_kind="uniform", lo=32768, hi=131072),
}


def rng(seed: int, stream: int) -> np.random.Generator:
    """Independent numpy generator for one stream of one workload seed."""
    return np.random.default_rng([seed, stream])


def context_lengths(w: Workload) -> np.ndarray:
    """Per-sequence context lengths (int64) drawn as the workload states.

    The 13B and 70B recipes use numpy's ``default_rng(seed)`` lognormal draw,
    rounded to the nearest integer and clipped; the long-context recipe draws
    integers uniformly in [lo, hi] inclusive.  These reproduce the batch sums
    24,860 (13B, seed 1), 451,896 (70B, seed 2) and 854,921 (long, seed 4).
    """
    if w.length_kind == "fixed":
        return np.asarray(w.fixed_lengths, dtype=np.int64)
    if w.length_kind == "lognormal":
        g = np.random.default_rng(w.seed)
        x = g.lognormal(np.log(w.median), w.sigma, w.num_seqs)
        return np.clip(np.rint(x), w.lo, w.hi).astype(np.int64)
    if w.length_kind == "uniform":
        g = np.random.default_rng(w.seed)
        return g.integers(w.lo, w.hi, w.num_seqs, endpoint=True).astype(np.int64)
    if w.length_kind == "prefix":
        suf = suffix_lengths(w)
        return (w.prompt_len + suf).astype(np.int64)
    raise ValueError(w.length_kind)


def suffix_lengths(w: Workload) -> np.ndarray:
    """Per-sample generated-suffix lengths of the shared-prefix workload."""
    g = rng(w.seed, STREAM_SUFFIX)
    n = w.num_prompts * w.samples_per_prompt
    return g.integers(w.suffix_lo, w.suffix_hi, n, endpoint=True).astype(np.int64)


def pool_order(num_blocks: int, seed: int) -> np.ndarray:
    """A seeded permutation of physical block ids (the order the free list hands them out)."""
    return rng(seed, STREAM_POOL_ORDER).permutation(num_blocks).astype(np.int32)


def normal_host(shape, seed: int, stream: int) -> np.ndarray:
    """N(0,1) draws as float32 on the host (small tensors only)."""
    return rng(seed, stream).standard_normal(size=shape, dtype=np.float32)


_TORCH_DTYPES = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}


def torch_dtype(name: str):
    import torch
    return getattr(torch, _TORCH_DTYPES[name])


def normal_tensor(shape, dtype: str, seed: int, stream: int, device: str = "cpu"):
    """N(0,1) draws rounded to ``dtype``, produced by torch's seeded generator on ``device``.

    Large pools are drawn on the device they will live on; the same call with the
    same seed and device always returns the same values.
    """
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 1000003 + int(stream))
    x = torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32)
    return x.to(torch_dtype(dtype))


def fill_normal_(t, seed: int, stream: int, chunk_rows: int = 4096):
    """Fill an existing tensor with N(0,1) draws in place, chunked along dim 0
    so that a multi-GB pool never needs a float32 staging copy of its full size."""
    import torch
    gen = torch.Generator(device=t.device)
    gen.manual_seed(int(seed) * 1000003 + int(stream))
    n = t.shape[0]
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        x = torch.randn((r1 - r0,) + tuple(t.shape[1:]), generator=gen, device=t.device,
                        dtype=torch.float32)
        t[r0:r1].copy_(x)
    return t


def fp8_scales(num_kv_heads: int, seed: int) -> np.ndarray:
    """Per-KV-head fp32 scales for an fp8 cache of N(0,1) data: a seeded value in
    [3, 6] / 448 per head, so that 3 to 6 standard deviations reach the largest
    E4M3 magnitude."""
    return (rng(seed, STREAM_SCALES).uniform(3.0, 6.0, num_kv_heads) / 448.0).astype(np.float32)


def fill_fp8_codes_(t, scales, seed: int, stream: int, chunk_rows: int = 4096):
    """Fill a uint8 fp8 cache ([NB, Hkv, ...], head axis 1) with the E4M3 codes of
    N(0,1) draws divided by the head's scale and clipped to +-448, chunked along
    dim 0.  The codes come from torch's float8_e4m3fn cast of the draws: synthetic
    input only (never a NaN code)."""
    import torch
    gen = torch.Generator(device=t.device)
    gen.manual_seed(int(seed) * 1000003 + int(stream))
    inv = (1.0 / torch.as_tensor(np.asarray(scales, dtype=np.float32), device=t.device))
    inv = inv.view((1, -1) + (1,) * (t.dim() - 2))
    n = t.shape[0]
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        x = torch.randn((r1 - r0,) + tuple(t.shape[1:]), generator=gen, device=t.device,
                        dtype=torch.float32)
        t[r0:r1].copy_((x * inv).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8))
    return t


def int8_scales(num_kv_heads: int, seed: int) -> np.ndarray:
    """Per-KV-head fp32 scales for an int8 cache of N(0,1) data: a seeded value in
    [3, 6] / 127 per head, so that 3 to 6 standard deviations reach code 127."""
    return (rng(seed, STREAM_SCALES).uniform(3.0, 6.0, num_kv_heads) / 127.0).astype(np.float32)


def fill_int8_codes_(t, scales, seed: int, stream: int, chunk_rows: int = 4096):
    """Fill an int8 cache ([NB, Hkv, ...], head axis 1) with N(0,1) draws divided
    by the head's scale, rounded by torch and clipped to +-127, chunked along
    dim 0: synthetic input only."""
    import torch
    gen = torch.Generator(device=t.device)
    gen.manual_seed(int(seed) * 1000003 + int(stream))
    inv = (1.0 / torch.as_tensor(np.asarray(scales, dtype=np.float32), device=t.device))
    inv = inv.view((1, -1) + (1,) * (t.dim() - 2))
    n = t.shape[0]
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        x = torch.randn((r1 - r0,) + tuple(t.shape[1:]), generator=gen, device=t.device,
                        dtype=torch.float32)
        t[r0:r1].copy_((x * inv).round_().clamp_(-127.0, 127.0).to(torch.int8))
    return t


def describe(w: Workload, lengths: Optional[np.ndarray] = None) -> dict:
    lengths = context_lengths(w) if lengths is None else lengths
    return {
        "workload": w.name, "num_seqs": int(len(lengths)), "num_q_heads": w.num_q_heads,
        "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "dtype": w.dtype,
        "block_size": w.block_size, "sum_context": int(lengths.sum()),
        "max_context": int(lengths.max()), "seed": w.seed,
    }

"""Decode batches for the GPU parity tests.

Tables and slots come from the oracle's block manager; values come from the
shared seeded generators.  The oracle's copy of the cache is taken from the
generator's output before any library kernel touches the device copy, and the
oracle applies its own cache write to it, so no oracle input ever comes from
the CUDA path.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

from oracle import cache_ops, paged_attention
from oracle.block_manager import BlockManager
from paged_kv_cache_166_gb300 import workloads as W


@dataclasses.dataclass
class Batch:
    w: W.Workload
    lens: np.ndarray
    NB: int
    tables: np.ndarray       # [S, MAXB] int32
    ctx: np.ndarray          # [S] int32
    new_slots: np.ndarray    # [S] int32 (slot of each sequence's new token)
    kc: torch.Tensor         # device caches, before the new tokens are written
    vc: torch.Tensor
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor

    def device_index(self, dev):
        return (torch.from_numpy(self.tables).to(dev), torch.from_numpy(self.ctx).to(dev),
                torch.from_numpy(self.new_slots).to(dev))


def blocks_needed(lens, B) -> int:
    return int(sum(-(-int(t) // B) for t in lens))


def decode_batch(w: W.Workload, lens: Optional[np.ndarray] = None, device="cuda",
                 pool_blocks: Optional[int] = None, maxb_extra: int = 0) -> Batch:
    """History of ctx-1 tokens per sequence, then one new token each (write-then-attend)."""
    lens = W.context_lengths(w) if lens is None else np.asarray(lens, dtype=np.int64)
    S, B = len(lens), w.block_size
    NB = pool_blocks or w.fixed_pool_blocks or int(np.ceil(blocks_needed(lens, B) * (1 + w.pool_spare))) + 1
    mgr = BlockManager(NB, B, W.pool_order(NB, w.seed))
    sids = [mgr.create() for _ in range(S)]
    for s, t in zip(sids, lens):
        if t > 0:
            mgr.append(s, int(t) - 1)
    new_slots = np.full(S, -1, dtype=np.int32)
    for i, (s, t) in enumerate(zip(sids, lens)):
        if t > 0:
            new_slots[i] = mgr.append(s, 1)[0][0]
    maxb = max(1, max(len(mgr.tables[s]) for s in sids)) + maxb_extra
    tables, ctx = mgr.export_tables(sids, maxb)
    shape = (NB, w.num_kv_heads, B, w.head_dim)
    kc = torch.empty(shape, dtype=W.torch_dtype(w.dtype), device=device)
    vc = torch.empty_like(kc)
    W.fill_normal_(kc, w.seed, W.STREAM_K_POOL)
    W.fill_normal_(vc, w.seed, W.STREAM_V_POOL)
    q = W.normal_tensor((S, w.num_q_heads, w.head_dim), w.dtype, w.seed, W.STREAM_Q, device)
    kn = W.normal_tensor((S, w.num_kv_heads, w.head_dim), w.dtype, w.seed, W.STREAM_K_NEW, device)
    vn = W.normal_tensor((S, w.num_kv_heads, w.head_dim), w.dtype, w.seed, W.STREAM_V_NEW, device)
    return Batch(w, lens, NB, tables, ctx, new_slots, kc, vc, q, kn, vn)


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def oracle_rows(b: Batch, seqs: List[int]) -> np.ndarray:
    """fp64 oracle output rows [len(seqs), Hq, D] of the listed sequences.

    Gathers only the blocks those sequences use (from the caches as generated),
    relabels them compactly (the oracle is invariant to physical ids), applies the
    oracle cache write of the sequences' new tokens, then runs the oracle.
    Must be called before the device caches are written by the library.
    """
    B = b.w.block_size
    used = sorted({int(x) for s in seqs for x in b.tables[s, :-(-int(b.ctx[s]) // B)]})
    remap = {old: i for i, old in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=b.kc.device)
    kc = np64(b.kc.index_select(0, idx)) if used else np.zeros((0,) + tuple(b.kc.shape[1:]))
    vc = np64(b.vc.index_select(0, idx)) if used else np.zeros((0,) + tuple(b.vc.shape[1:]))
    tables = np.zeros((len(seqs), b.tables.shape[1]), dtype=np.int32)
    ctx = np.zeros(len(seqs), dtype=np.int32)
    slots = np.full(len(seqs), -1, dtype=np.int32)
    for r, s in enumerate(seqs):
        nb = -(-int(b.ctx[s]) // B)
        tables[r, :nb] = [remap[int(x)] for x in b.tables[s, :nb]]
        ctx[r] = b.ctx[s]
        if b.new_slots[s] >= 0:
            old = int(b.new_slots[s])
            slots[r] = remap[old // B] * B + old % B
    sel = torch.tensor(seqs, dtype=torch.long, device=b.q.device)
    cache_ops.kv_write(np64(b.k_new.index_select(0, sel)), np64(b.v_new.index_select(0, sel)),
                       slots, kc, vc)
    return paged_attention.paged_attention(np64(b.q.index_select(0, sel)), kc, vc, tables, ctx,
                                           b.w.scale)


def row_errors(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """max_d |got - ref| / ||ref_row||_2 per (sequence, head) row (zero rows: absolute)."""
    err = np.abs(got - ref).max(axis=-1)
    norm = np.linalg.norm(ref, axis=-1)
    return np.where(norm > 0, err / np.where(norm > 0, norm, 1), err)


def tolerance(dtype: str) -> float:
    """Row tolerance: 1e-5 for fp32, 2e-3 for fp16/bf16 (fp32 accumulation)."""
    return 1e-5 if dtype == "f32" else 2e-3

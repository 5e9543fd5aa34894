"""GPU parity of preemption by swapping against the oracle.

A sequence's blocks go to page-locked host memory and come back into freshly
allocated blocks ("PagedAttention — how vLLM stopped wasting 80% of your GPU
memory", section "Preemption: what happens when memory runs out anyway"):

* the host buffers hold exactly the oracle's copies of the blocks (bytes
  compared), for 16-bit and fp8 caches;
* the library's block manager hands out the same ids as the oracle's on
  swap-out and swap-in;
* after the released blocks are overwritten with NaN and the sequence is
  swapped back in, decode attention over the batch is bit-identical to before
  the swap, and matches the oracle;
* host memory the device cannot address is refused before any work is queued.
"""
import ctypes

import numpy as np
import pytest
import torch

import batches as BT
from oracle import cache_ops
from oracle.block_manager import BlockManager
from paged_kv_cache_166_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()


def pkv():
    import paged_kv_cache_166_gb300 as m
    return m


def test_swap_round_trip_matches_oracle_and_restores_attention():
    import dataclasses
    from paged_kv_cache_166_gb300 import BlockAllocator
    w = dataclasses.replace(W.WORKLOADS["gqa70b"], num_q_heads=16, num_kv_heads=2)
    lens = np.array([700, 33, 2048, 17, 1200, 5])
    B, S = 16, len(lens)
    NB = int(sum(-(-t // B) for t in lens)) + 40
    order = W.pool_order(NB, 5)
    lib, orc = BlockAllocator(NB, B, order), BlockManager(NB, B, order)
    sids = []
    for t in lens:
        a, o = lib.create(), orc.create()
        assert a == o
        lib.append(a, int(t))
        orc.append(o, int(t))
        sids.append(a)
    shape = (NB, w.num_kv_heads, B, w.head_dim)
    kc = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    W.fill_normal_(kc, 9, W.STREAM_K_POOL)
    W.fill_normal_(vc, 9, W.STREAM_V_POOL)
    okc, ovc = BT.np64(kc), BT.np64(vc)          # the oracle's copies
    q = W.normal_tensor((S, w.num_q_heads, w.head_dim), "bf16", 9, W.STREAM_Q, "cuda")

    def attend():
        tab, ctx = lib.export_tables(sids, 128)
        out = torch.full_like(q, float("nan"))
        pkv().paged_decode_attention(q, kc, vc, torch.from_numpy(tab).cuda(),
                                     torch.from_numpy(ctx).cuda(), w.scale, out)
        torch.cuda.synchronize()
        return out

    before = attend()
    victims = [2, 4]
    hosts = {}
    for v in victims:
        ids = lib.swap_out(sids[v])
        assert ids == orc.swap_out(sids[v])
        n = len(ids)
        hk = torch.empty((n,) + shape[1:], dtype=kc.dtype).pin_memory()
        hv = torch.empty_like(hk).pin_memory()
        pkv().paged_swap_out(kc, vc, torch.tensor(ids, dtype=torch.int32, device="cuda"), hk, hv)
        torch.cuda.synchronize()
        ok, ov = cache_ops.swap_out_blocks(okc, ovc, ids)
        assert np.array_equal(hk.to(torch.float64).numpy(), ok)
        assert np.array_equal(hv.to(torch.float64).numpy(), ov)
        hosts[v] = (hk, hv)
    # the released blocks are reused: fill every free block with NaN
    free = [b for b in range(NB) if lib.refcount(b) == 0]
    fi = torch.tensor(free, dtype=torch.long, device="cuda")
    kc.index_fill_(0, fi, float("nan"))
    vc.index_fill_(0, fi, float("nan"))
    okc[free] = np.nan
    ovc[free] = np.nan
    for v in victims[::-1]:
        new = lib.swap_in(sids[v])
        assert new == orc.swap_in(sids[v])
        hk, hv = hosts[v]
        pkv().paged_swap_in(hk, hv, torch.tensor(new, dtype=torch.int32, device="cuda"), kc, vc)
        cache_ops.swap_in_blocks(BT.np64(hk), BT.np64(hv), new, okc, ovc)
    torch.cuda.synchronize()
    assert np.array_equal(BT.np64(kc), okc, equal_nan=True)
    assert np.array_equal(BT.np64(vc), ovc, equal_nan=True)
    after = attend()
    assert torch.equal(before.view(torch.int16), after.view(torch.int16))
    tab, ctx = orc.export_tables(sids, 128)
    from oracle import paged_attention as pa
    ref = pa.paged_attention(BT.np64(q), okc, ovc, tab, ctx, w.scale)
    err = BT.row_errors(BT.np64(after), ref)
    assert err.max() <= BT.tolerance("bf16")


def test_swap_fp8_blocks_bytes_round_trip():
    NB, Hkv, D = 12, 2, 128
    kc = torch.randint(0, 255, (NB, Hkv, 16, D), dtype=torch.uint8, device="cuda")
    vc = torch.randint(0, 255, (NB, Hkv, D, 16), dtype=torch.uint8, device="cuda")
    k0, v0 = kc.clone(), vc.clone()
    ids = torch.tensor([7, 2, 11, 0], dtype=torch.int32, device="cuda")
    hk = torch.empty((4, Hkv, 16, D), dtype=torch.uint8).pin_memory()
    hv = torch.empty((4, Hkv, D, 16), dtype=torch.uint8).pin_memory()
    pkv().paged_swap_out(kc, vc, ids, hk, hv)
    torch.cuda.synchronize()
    assert torch.equal(hk, k0[ids.long()].cpu()) and torch.equal(hv, v0[ids.long()].cpu())
    new = torch.tensor([1, 3, 5, 9], dtype=torch.int32, device="cuda")
    pkv().paged_swap_in(hk, hv, new, kc, vc)
    torch.cuda.synchronize()
    assert torch.equal(kc[new.long()], k0[ids.long()]) and torch.equal(vc[new.long()], v0[ids.long()])


def test_swap_refuses_pageable_host_memory():
    from paged_kv_cache_166_gb300 import _native as N
    kc = torch.zeros((4, 1, 16, 64), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    ids = torch.tensor([1], dtype=torch.int32, device="cuda")
    pageable = torch.empty((1, 1, 16, 64), dtype=torch.float16)
    with pytest.raises(ValueError):
        pkv().paged_swap_out(kc, vc, ids, pageable, pageable)
    buf = np.zeros(16 * 64 * 2, dtype=np.uint8)       # plain (pageable) host memory
    ptr = buf.ctypes.data_as(ctypes.c_void_p)
    rc = N.lib().pkv_swap_out_blocks(kc.data_ptr(), vc.data_ptr(), ids.data_ptr(), 1, 4,
                                     16 * 64 * 2, ptr, ptr, torch.cuda.current_stream().cuda_stream)
    assert rc == N.PKV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert not buf.any()

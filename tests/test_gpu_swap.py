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
* host memory the device cannot address is refused before any work is queued;
* the all-layer calls move every layer's blocks to and from host block
  l * n + i exactly as one single-layer call per layer does.
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


def _raw(t):
    return (t.view(torch.int16) if t.element_size() == 2 else t).cpu().numpy()


@pytest.mark.parametrize("dtype,L", [(torch.float16, 3), (torch.bfloat16, 5), (torch.uint8, 2)])
def test_swap_layers_round_trip_matches_oracle(dtype, L):
    """Every layer's blocks go to host block l * n + i in one launch (bytes equal the
    oracle's per-layer copies and one single-layer call per layer); out-of-pool ids
    leave their host blocks alone; swapping back in to fresh ids restores every
    layer's blocks bit for bit and touches nothing else."""
    g = torch.Generator().manual_seed(40 + L)
    NB, Hkv, B, D = 16, 2, 16, 64
    if dtype == torch.uint8:
        make = lambda: torch.randint(0, 256, (NB, Hkv, B, D), generator=g, dtype=dtype)
    else:
        make = lambda: torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    kh = [make() for _ in range(L)]
    vh = [make() for _ in range(L)]
    kd = [t.cuda() for t in kh]
    vd = [t.cuda() for t in vh]
    ids_np = np.array([7, 2, -1, 11, 0], dtype=np.int32)
    n = len(ids_np)
    ids = torch.from_numpy(ids_np).cuda()
    bb = Hkv * B * D * kd[0].element_size()
    hk = torch.full((L * n * bb,), 0x5A, dtype=torch.uint8).pin_memory()
    hv = torch.full((L * n * bb,), 0x5A, dtype=torch.uint8).pin_memory()
    pkv().paged_swap_out_layers(kd, vd, ids, hk, hv)
    # the same through one single-layer call per layer
    sk = [torch.full((n * bb,), 0x5A, dtype=torch.uint8).pin_memory() for _ in range(L)]
    sv = [torch.full((n * bb,), 0x5A, dtype=torch.uint8).pin_memory() for _ in range(L)]
    for l in range(L):
        pkv().paged_swap_out(kd[l], vd[l], ids, sk[l], sv[l])
    torch.cuda.synchronize()
    valid = ids_np >= 0
    for l in range(L):
        ok_, ov_ = cache_ops.swap_out_blocks(_raw(kh[l]), _raw(vh[l]), ids_np[valid])
        hk_l = hk[l * n * bb:(l + 1) * n * bb].numpy().reshape(n, bb)
        hv_l = hv[l * n * bb:(l + 1) * n * bb].numpy().reshape(n, bb)
        assert np.array_equal(hk_l[valid], ok_.reshape(valid.sum(), -1).view(np.uint8))
        assert np.array_equal(hv_l[valid], ov_.reshape(valid.sum(), -1).view(np.uint8))
        assert (hk_l[~valid] == 0x5A).all() and (hv_l[~valid] == 0x5A).all()
        assert torch.equal(hk[l * n * bb:(l + 1) * n * bb], sk[l])
        assert torch.equal(hv[l * n * bb:(l + 1) * n * bb], sv[l])
    # back in, to fresh ids (the out-of-pool entry stays skipped)
    new_np = np.array([1, 3, -1, 5, 9], dtype=np.int32)
    for t in kd + vd:
        t[torch.from_numpy(new_np[valid]).long().cuda()] = 0
    pkv().paged_swap_in_layers(hk, hv, torch.from_numpy(new_np).cuda(), kd, vd)
    torch.cuda.synchronize()
    for l in range(L):
        for src_h, got in ((kh[l], kd[l]), (vh[l], vd[l])):
            want = _raw(src_h).copy()
            want[new_np[valid]] = _raw(src_h)[ids_np[valid]]
            assert np.array_equal(_raw(got), want)


def test_swap_layers_refusals():
    from paged_kv_cache_166_gb300 import _native as N
    kc = [torch.zeros((4, 1, 16, 64), dtype=torch.float16, device="cuda") for _ in range(129)]
    ids = torch.tensor([1], dtype=torch.int32, device="cuda")
    bb = 16 * 64 * 2
    pinned = torch.empty((129 * bb,), dtype=torch.uint8).pin_memory()
    with pytest.raises(pkv().PkvError):
        pkv().paged_swap_out_layers(kc, kc, ids, pinned, pinned)     # more than 128 layers
    pageable = torch.empty((2 * bb,), dtype=torch.uint8)
    with pytest.raises(ValueError):
        pkv().paged_swap_out_layers(kc[:2], kc[2:4], ids, pageable, pageable)
    with pytest.raises(ValueError):                                  # too small for 3 layers
        pkv().paged_swap_in_layers(pinned[:2 * bb], pinned[:2 * bb], ids, kc[:3], kc[3:6])
    buf = np.zeros(2 * bb, dtype=np.uint8)                           # plain host memory
    ptr = buf.ctypes.data_as(ctypes.c_void_p)
    kp = (ctypes.c_void_p * 2)(kc[0].data_ptr(), kc[1].data_ptr())
    vp = (ctypes.c_void_p * 2)(kc[2].data_ptr(), kc[3].data_ptr())
    rc = N.lib().pkv_swap_out_blocks_layers(kp, vp, 2, ids.data_ptr(), 1, 4, bb, ptr, ptr,
                                            torch.cuda.current_stream().cuda_stream)
    assert rc == N.PKV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert not buf.any()

"""Shared-prefix parallel sampling on the GPU: 32 prompts x 8 samples.

Each prompt of 1,000 tokens is written once; its 8 samples share the prompt
blocks through refcounts, the first write into the shared partial last block
triggers copy-on-write, and each sample appends a suffix of 0..512 tokens
("PagedAttention and vLLM: Virtual Memory for the KV Cache", "A second
calculation: parallel sampling with block sharing"; "PagedAttention: How vLLM
Borrowed Virtual Memory...", section "Copy-on-Write for Beam Search and Parallel
Sampling").  Device order: cache write of the prompts, the copy-on-write block
copies, the cache write of the suffixes, then decode attention.

Checks: the library's block manager issues the same tables, slots and copy pairs
as the oracle's; the device caches equal the oracle's caches bit for bit;
sampled attention rows match the oracle; and attention over the shared layout
is bit-identical to attention over a layout where every sample owns private
copies of its prompt blocks (same data, same lengths).
"""
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


def build_shared(w, num_prompts, samples, lens_suffix, make_mgr, NB):
    mgr = make_mgr(NB)
    P, B = w.prompt_len, w.block_size
    prompt_slots, suffix_slots, cows, seqs = [], [], [], []
    for p in range(num_prompts):
        parent = mgr.create()
        prompt_slots.append(np.asarray(mgr.append(parent, P)[0], dtype=np.int32))
        group = [parent] + [mgr.fork(parent) for _ in range(samples - 1)]
        for i, sid in enumerate(group):
            sl, cw = mgr.append(sid, int(lens_suffix[p * samples + i]))
            suffix_slots.append(np.asarray(sl, dtype=np.int32))
            cows.extend(cw)
        seqs.extend(group)
    return mgr, seqs, np.concatenate(prompt_slots), np.concatenate(suffix_slots), cows


def test_shared_prefix_full_workload():
    import paged_kv_cache_166_gb300 as pkv
    w = W.WORKLOADS["prefix"]
    B, P = w.block_size, w.prompt_len
    nprompt, nsamp = w.num_prompts, w.samples_per_prompt
    suf = W.suffix_lengths(w)
    ctx_all = P + suf
    # full prompt blocks once per prompt, plus each sample's own blocks (upper bound)
    blocks = nprompt * (P // B) + sum(-(-int(t) // B) - P // B for t in ctx_all)
    NB = int(blocks * 1.1) + 8
    order = W.pool_order(NB, w.seed)

    mgr, seqs, pslots, sslots, cows = build_shared(
        w, nprompt, nsamp, suf, lambda nb: BlockManager(nb, B, order), NB)
    lib_mgr, lseqs, lp, ls, lc = build_shared(
        w, nprompt, nsamp, suf, lambda nb: pkv.BlockAllocator(nb, B, order), NB)
    assert lseqs == seqs and np.array_equal(lp, pslots) and np.array_equal(ls, sslots)
    assert lc == cows and 0 < len(cows) <= nprompt * (nsamp - 1)
    maxb = max(len(mgr.tables[s]) for s in seqs)
    tables, ctx = mgr.export_tables(seqs, maxb)
    lt, lctx = lib_mgr.export_tables(lseqs, maxb)
    assert np.array_equal(lt, tables) and np.array_equal(lctx, ctx)
    assert NB - mgr.num_free() < nprompt * nsamp * (-(-P // B))   # sharing saves blocks

    dt = W.torch_dtype(w.dtype)
    Hkv, D = w.num_kv_heads, w.head_dim
    kp = W.normal_tensor((len(pslots), Hkv, D), w.dtype, w.seed, W.STREAM_K_NEW, "cuda")
    vp = W.normal_tensor((len(pslots), Hkv, D), w.dtype, w.seed, W.STREAM_V_NEW, "cuda")
    ks = W.normal_tensor((len(sslots), Hkv, D), w.dtype, w.seed + 100, W.STREAM_K_NEW, "cuda")
    vs = W.normal_tensor((len(sslots), Hkv, D), w.dtype, w.seed + 100, W.STREAM_V_NEW, "cuda")
    q = W.normal_tensor((len(seqs), w.num_q_heads, D), w.dtype, w.seed, W.STREAM_Q, "cuda")
    kc = torch.full((NB, Hkv, B, D), float("nan"), dtype=dt, device="cuda")
    vc = torch.full_like(kc, float("nan"))

    # oracle caches (host, fp32 holds bf16 exactly)
    kh = np.full(kc.shape, np.nan, dtype=np.float32)
    vh = np.full(kc.shape, np.nan, dtype=np.float32)
    cache_ops.kv_write(kp.float().cpu().numpy(), vp.float().cpu().numpy(), pslots, kh, vh)
    cache_ops.copy_blocks(kh, vh, cows)
    cache_ops.kv_write(ks.float().cpu().numpy(), vs.float().cpu().numpy(), sslots, kh, vh)

    # device: same order through the library
    pkv.paged_kv_write(kp, vp, torch.from_numpy(pslots).cuda(), kc, vc)
    pkv.paged_copy_blocks(kc, vc, torch.tensor(cows, dtype=torch.int32).cuda())
    pkv.paged_kv_write(ks, vs, torch.from_numpy(sslots).cuda(), kc, vc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(kc.float().cpu().numpy(), kh)
    np.testing.assert_array_equal(vc.float().cpu().numpy(), vh)

    td, cd = torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda()
    out = torch.empty_like(q)
    pkv.paged_decode_attention(q, kc, vc, td, cd, w.scale, out)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    pick = sorted({int(np.argmax(ctx)), int(np.argmin(ctx))} |
                  set(rng.choice(len(seqs), 16, replace=False).tolist()))
    from oracle import paged_attention
    ref = paged_attention.paged_attention(q.double().cpu().numpy()[pick], kh, vh, tables[pick],
                                          ctx[pick], w.scale)
    err = BT.row_errors(out.double().cpu().numpy()[pick], ref)
    assert err.max() <= BT.tolerance(w.dtype), err.max()

    # private copies: every sample owns a copy of every prompt block
    priv = pkv.BlockAllocator(NB + nprompt * nsamp * (-(-P // B)), B)
    NBp = priv.num_blocks
    kc2 = torch.full((NBp, Hkv, B, D), float("nan"), dtype=dt, device="cuda")
    vc2 = torch.full_like(kc2, float("nan"))
    pseqs, all_slots, src_rows = [], [], []
    pos_suffix = 0
    for p in range(nprompt):
        for i in range(nsamp):
            sid = priv.create()
            n = int(suf[p * nsamp + i])
            sl, cw = priv.append(sid, P + n)
            assert cw == []
            all_slots.append(sl)
            src_rows.append(("p", p * P, P))
            src_rows.append(("s", pos_suffix, n))
            pos_suffix += n
            pseqs.append(sid)
    k_rows = torch.cat([(kp if kind == "p" else ks)[a:a + n] for kind, a, n in src_rows])
    v_rows = torch.cat([(vp if kind == "p" else vs)[a:a + n] for kind, a, n in src_rows])
    slots2 = torch.from_numpy(np.concatenate(all_slots).astype(np.int32)).cuda()
    pkv.paged_kv_write(k_rows.contiguous(), v_rows.contiguous(), slots2, kc2, vc2)
    t2, c2 = priv.export_tables(pseqs, maxb)
    assert np.array_equal(c2, ctx)
    out2 = torch.empty_like(q)
    pkv.paged_decode_attention(q, kc2, vc2, torch.from_numpy(t2).cuda(), torch.from_numpy(c2).cuda(),
                               w.scale, out2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)

"""GPU parity of decode attention and the decode step for cache block sizes 8
and 32 (the pages' tuning knob: "Different workloads ... can benefit from
tuning it", "PagedAttention — how vLLM stopped wasting 80% of your GPU memory",
FAQ "Why 16 tokens per block specifically?").

The kernels compute in 16-token steps whatever the block size: a step reads
half of a 32-token block, or two 8-token blocks.  Covered: reduced workload
shapes under several warp counts, every row against the oracle; edge lengths
around 8/16/32 with NaN in every slot past a context and in unused blocks; the
decode step bit-identical to the write followed by the attention; and the same
logical data laid out with block sizes 8, 16 and 32 giving bit-identical
outputs (the 16-token step schedule does not depend on the block size).
"""
import dataclasses

import numpy as np
import pytest
import torch

import batches as BT
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


def run(b, num_warps=0):
    tables, ctx, slots = b.device_index("cuda")
    pkv().paged_kv_write(b.k_new, b.v_new, slots, b.kc, b.vc)
    out = torch.full_like(b.q, float("nan"))
    pkv().paged_decode_attention(b.q, b.kc, b.vc, tables, ctx, b.w.scale, out, num_warps=num_warps)
    torch.cuda.synchronize()
    return out


def check(b, seqs, got, ref):
    err = BT.row_errors(BT.np64(got)[seqs], ref)
    assert err.max() <= BT.tolerance(b.w.dtype), f"row error {err.max():.3e}"


CASES = [
    ("mha13b", dict(num_q_heads=8, num_kv_heads=8), (300, 1, 2048, 77, 16, 513, 129, 31)),
    ("gqa70b", dict(num_q_heads=32, num_kv_heads=4), (1024, 5, 3000, 16, 17, 700, 1, 2100)),
    ("longctx", dict(num_q_heads=16, num_kv_heads=2), (9000, 4097)),
]


@pytest.mark.parametrize("B", [8, 32])
@pytest.mark.parametrize("name,kw,lens", CASES)
@pytest.mark.parametrize("num_warps", [0, 3, 61])
def test_block_size_every_row(B, name, kw, lens, num_warps):
    w = dataclasses.replace(W.WORKLOADS[name], block_size=B, **kw)
    b = BT.decode_batch(w, np.asarray(lens))
    seqs = list(range(len(lens)))
    ref = BT.oracle_rows(b, seqs)
    check(b, seqs, run(b, num_warps), ref)


@pytest.mark.parametrize("B", [8, 32])
@pytest.mark.parametrize("dtype,D,G", [("bf16", 128, 8), ("f16", 128, 1), ("bf16", 64, 4)])
def test_block_size_edge_lengths_with_nan(B, dtype, D, G):
    w = dataclasses.replace(W.WORKLOADS["tiny"], dtype=dtype, head_dim=D, num_kv_heads=2,
                            num_q_heads=2 * G, fixed_pool_blocks=0, seed=23, block_size=B)
    lens = np.array([0, 1, 7, 8, 9, 15, 16, 17, 31, 32, 33, 40 * B // 8])
    b = BT.decode_batch(w, lens, maxb_extra=0)
    for s, t in enumerate(lens):
        if t % B:
            blk = int(b.tables[s, (t - 1) // B])
            b.kc[blk, :, t % B:, :] = float("nan")
            b.vc[blk, :, t % B:, :] = float("nan")
    used = {int(x) for s, t in enumerate(lens) for x in b.tables[s, :-(-int(t) // B)]}
    unused = torch.tensor([i for i in range(b.NB) if i not in used], dtype=torch.long, device="cuda")
    if len(unused):
        b.kc[unused] = float("nan")
        b.vc[unused] = float("nan")
    seqs = list(range(len(lens)))
    ref = BT.oracle_rows(b, seqs)
    got = run(b)
    assert torch.isfinite(got).all()
    check(b, seqs, got, ref)


@pytest.mark.parametrize("B", [8, 32])
def test_block_size_decode_step_equals_write_then_attend(B):
    w = dataclasses.replace(W.WORKLOADS["gqa70b"], num_q_heads=16, num_kv_heads=2, block_size=B)
    lens = np.array([700, 1, 33, 2048, 16, 9, 900])
    a = BT.decode_batch(w, lens)
    c = BT.decode_batch(w, lens)
    out_a = run(a)
    tables, ctx, _ = c.device_index("cuda")
    out_c = torch.full_like(c.q, float("nan"))
    pkv().paged_decode_step(c.q, c.k_new, c.v_new, c.kc, c.vc, tables, ctx, w.scale, out_c)
    torch.cuda.synchronize()
    assert torch.equal(a.kc, c.kc) and torch.equal(a.vc, c.vc)
    assert torch.equal(out_a.view(torch.int16), out_c.view(torch.int16))


def test_outputs_do_not_depend_on_block_size():
    """The same logical K/V under block sizes 8, 16, 32: bit-identical outputs."""
    from paged_kv_cache_166_gb300 import BlockAllocator
    lens = [1, 8, 9, 16, 17, 33, 130, 700]
    Hq, Hkv, D = 16, 2, 128
    kv = [W.normal_tensor((t, Hkv, D), "bf16", 31, W.STREAM_K_NEW, "cuda") for t in lens]
    vv = [W.normal_tensor((t, Hkv, D), "bf16", 31, W.STREAM_V_NEW, "cuda") for t in lens]
    q = W.normal_tensor((len(lens), Hq, D), "bf16", 31, W.STREAM_Q, "cuda")
    outs = []
    for B in (8, 16, 32):
        NB = sum(-(-t // B) for t in lens) + 3
        al = BlockAllocator(NB, B, W.pool_order(NB, B))
        sids = [al.create() for _ in lens]
        kc = torch.zeros((NB, Hkv, B, D), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        for s, t, k, v in zip(sids, lens, kv, vv):
            slots, _ = al.append(s, t)
            pkv().paged_kv_write(k, v, torch.from_numpy(slots).cuda(), kc, vc)
        tab, ctx = al.export_tables(sids, -(-max(lens) // B))
        out = torch.empty_like(q)
        pkv().paged_decode_attention(q, kc, vc, torch.from_numpy(tab).cuda(),
                                     torch.from_numpy(ctx).cuda(), 0.088, out)
        torch.cuda.synchronize()
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[2].view(torch.int16), outs[1].view(torch.int16))

"""GPU parity of paged decode attention against the fp64 oracle.

Row tolerance (max over d of |gpu - oracle| divided by the oracle row's L2
norm): 1e-5 for fp32, 2e-3 for fp16/bf16.  Covered:

* all five workload shapes, reduced so the oracle checks every row, under
  several worker-warp counts so that contexts are cut into 1..many pieces;
* the full-size 13B, 70B and long-context batches in the launch configuration
  bench.py times (default warps), every row (13B) or sampled rows;
* edge cases: empty contexts, lengths 1/15/16/17/31/32/33 and a full table, NaN
  in every unused slot, all group sizes, head dims and dtypes;
* bit-identity under relabelling of physical blocks and between runs; reuse of
  one workspace across launches;
* invalid device data flagged in the status word without a fault;
* the decode step (the write of each new token, then the attention, chained in
  one call): bit-identical to the write followed by the attention (output and
  caches), and against the oracle, invalid device data included.
"""
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


def run(b: BT.Batch, num_warps=0, write=True):
    tables, ctx, slots = b.device_index("cuda")
    if write:
        pkv().paged_kv_write(b.k_new, b.v_new, slots, b.kc, b.vc)
    out = torch.full_like(b.q, float("nan"))
    pkv().paged_decode_attention(b.q, b.kc, b.vc, tables, ctx, b.w.scale, out,
                                 num_warps=num_warps)
    torch.cuda.synchronize()
    return out


def check_rows(b, seqs, got, ref):
    err = BT.row_errors(BT.np64(got)[seqs], ref)
    tol = BT.tolerance(b.w.dtype)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, f"row error {err.max():.3e} > {tol} at {worst}"
    return err.max()


def reduced(name, lens, **kw):
    import dataclasses
    w = dataclasses.replace(W.WORKLOADS[name], **kw)
    return w, np.asarray(lens)


REDUCED = {
    "tiny": reduced("tiny", (1, 17, 40, 100)),
    "mha13b": reduced("mha13b", (300, 1, 2048, 77, 16, 513, 129, 31)),
    "gqa70b": reduced("gqa70b", (1024, 5, 3000, 16, 17, 700, 1, 2100, 64, 250)),
    "prefix_shape": reduced("prefix", (1000, 1001, 1512, 1008), length_kind="fixed"),
    "longctx": reduced("longctx", (9000, 4097)),
}


@pytest.mark.parametrize("name", list(REDUCED))
@pytest.mark.parametrize("num_warps", [0, 1, 3, 16, 61])
def test_reduced_workloads_every_row(name, num_warps):
    w, lens = REDUCED[name]
    b = BT.decode_batch(w, lens)
    seqs = list(range(len(lens)))
    ref = BT.oracle_rows(b, seqs)
    got = run(b, num_warps)
    check_rows(b, seqs, got, ref)
    dev = torch.device("cuda", torch.cuda.current_device())
    m = pkv()
    ws = m.get_workspace(dev, w.group, w.head_dim, num_warps,
                         m.workspace_bytes(w.num_q_heads, w.num_kv_heads, w.head_dim, b.q.dtype,
                                           num_warps))
    assert m.decode_status(ws) == 0


def test_full_mha13b_every_row():
    b = BT.decode_batch(W.WORKLOADS["mha13b"])
    seqs = list(range(len(b.lens)))
    ref = BT.oracle_rows(b, seqs)
    check_rows(b, seqs, run(b), ref)


def sample(lens, k, seed):
    r = np.random.default_rng(seed)
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    pick |= set(r.choice(len(lens), size=min(k, len(lens)), replace=False).tolist())
    return sorted(pick)


def test_full_gqa70b_sampled_rows():
    b = BT.decode_batch(W.WORKLOADS["gqa70b"])
    seqs = sample(b.lens, 24, 0)
    ref = BT.oracle_rows(b, seqs)
    check_rows(b, seqs, run(b), ref)


def test_full_longctx_sampled_rows():
    b = BT.decode_batch(W.WORKLOADS["longctx"])
    seqs = sample(b.lens, 1, 1)
    ref = BT.oracle_rows(b, seqs)
    check_rows(b, seqs, run(b), ref)


@pytest.mark.parametrize("dtype,D,G", [
    ("bf16", 64, 1), ("bf16", 128, 2), ("bf16", 256, 4), ("f16", 64, 8), ("f16", 128, 4),
    ("f16", 256, 1), ("f32", 32, 8), ("f32", 64, 2), ("f32", 128, 1),
])
def test_edge_lengths_group_sizes_head_dims(dtype, D, G):
    import dataclasses
    w = dataclasses.replace(W.WORKLOADS["tiny"], dtype=dtype, head_dim=D, num_kv_heads=3,
                            num_q_heads=3 * G, fixed_pool_blocks=0, seed=17)
    lens = np.array([0, 1, 15, 16, 17, 31, 32, 33, 0, 160, 2])
    b = BT.decode_batch(w, lens, maxb_extra=0)
    # NaN in every slot no context reaches: a kernel that reads past a context fails
    B = w.block_size
    for s, t in enumerate(lens):
        if t % B:
            b.kc[int(b.tables[s, (t - 1) // B]), :, t % B:, :] = float("nan")
            b.vc[int(b.tables[s, (t - 1) // B]), :, t % B:, :] = float("nan")
    used = {int(x) for s, t in enumerate(lens) for x in b.tables[s, :-(-int(t) // B)]}
    unused = torch.tensor([i for i in range(b.NB) if i not in used], dtype=torch.long, device="cuda")
    b.kc[unused] = float("nan")
    b.vc[unused] = float("nan")
    seqs = list(range(len(lens)))
    ref = BT.oracle_rows(b, seqs)
    for nw in (0, 2, 7):
        got = run(b, nw, write=(nw == 0))
        check_rows(b, seqs, got, ref)
        assert torch.all(got[torch.from_numpy(lens == 0).cuda()] == 0)


def relabel(b: BT.Batch, seed: int) -> BT.Batch:
    """Same logical data under a random relabelling of physical blocks."""
    perm = np.random.default_rng(seed).permutation(b.NB)   # new id of block i = perm[i]
    inv = torch.from_numpy(np.argsort(perm)).cuda()
    import dataclasses
    return dataclasses.replace(
        b, kc=b.kc.index_select(0, inv), vc=b.vc.index_select(0, inv),
        tables=perm[b.tables].astype(np.int32),
        new_slots=np.where(b.new_slots >= 0, perm[np.maximum(b.new_slots, 0) // 16] * 16 + b.new_slots % 16,
                           -1).astype(np.int32))


@pytest.mark.parametrize("name", ["mha13b", "gqa70b"])
def test_physical_relabelling_is_bit_identical(name):
    w, lens = REDUCED[name]
    b = BT.decode_batch(w, lens)
    b2 = relabel(b, 5)
    out1 = run(b)
    out2 = run(b2)
    assert torch.equal(out1, out2)
    out3 = run(b, write=False)
    assert torch.equal(out1, out3)          # run to run


def test_warp_counts_agree_and_workspace_is_reusable():
    """Different cut points give the same rows within tolerance; a workspace used
    by one launch serves the next (the merge tickets are left at zero)."""
    w, lens = REDUCED["gqa70b"]
    b = BT.decode_batch(w, lens)
    ref = BT.oracle_rows(b, list(range(len(lens))))
    base = run(b, 0)
    m = pkv()
    ws = torch.zeros(m.workspace_bytes(w.num_q_heads, w.num_kv_heads, w.head_dim, b.q.dtype, 16),
                     dtype=torch.uint8, device="cuda")
    tables, ctx, _ = b.device_index("cuda")
    outs = []
    for _ in range(3):
        out = torch.full_like(b.q, float("nan"))
        m.paged_decode_attention(b.q, b.kc, b.vc, tables, ctx, w.scale, out, ws, 16)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    check_rows(b, list(range(len(lens))), base, ref)
    check_rows(b, list(range(len(lens))), outs[0], ref)
    tickets = ws[256:256 + 4 * 16].view(torch.int32)
    assert torch.count_nonzero(tickets) == 0


def test_invalid_device_data_is_flagged_not_faulted():
    m = pkv()
    w, lens = REDUCED["mha13b"]
    b = BT.decode_batch(w, lens)
    tables, ctx, slots = b.device_index("cuda")
    out = torch.empty_like(b.q)
    ws = torch.zeros(m.workspace_bytes(w.num_q_heads, w.num_kv_heads, w.head_dim, b.q.dtype),
                     dtype=torch.uint8, device="cuda")
    bad_ctx = ctx.clone()
    bad_ctx[2] = tables.shape[1] * 16 + 5           # longer than the table can hold
    bad_ctx[3] = -4
    m.paged_decode_attention(b.q, b.kc, b.vc, tables, bad_ctx, w.scale, out, ws)
    assert m.decode_status(ws) & 1
    assert torch.all(out[3] == 0) and torch.isfinite(out[2]).all()
    bad_tab = tables.clone()
    bad_tab[0, 0] = b.NB + 1000                    # outside the pool
    m.paged_decode_attention(b.q, b.kc, b.vc, bad_tab, ctx, w.scale, out, ws)
    assert m.decode_status(ws) & 2
    m.paged_decode_attention(b.q, b.kc, b.vc, tables, ctx, w.scale, out, ws)
    assert m.decode_status(ws) == 0
    # the same workspace under another warp count: flagged (zero-fill first to reuse)
    big = torch.zeros(m.workspace_bytes(w.num_q_heads, w.num_kv_heads, w.head_dim, b.q.dtype, 12),
                      dtype=torch.uint8, device="cuda")
    m.paged_decode_attention(b.q, b.kc, b.vc, tables, ctx, w.scale, out, big, 12)
    assert m.decode_status(big) == 0
    m.paged_decode_attention(b.q, b.kc, b.vc, tables, ctx, w.scale, out, big, 8)
    assert m.decode_status(big) & 8


def test_host_side_rejections():
    m = pkv()
    q = torch.zeros(2, 6, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 4, 16, 128, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(2, 2, dtype=torch.int32, device="cuda")
    c = torch.ones(2, dtype=torch.int32, device="cuda")
    with pytest.raises(m.PkvError):          # 6 query heads over 4 KV heads
        m.paged_decode_attention(q, kc, kc, t, c, 0.1, torch.empty_like(q))
    q2 = torch.zeros(2, 12, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.PkvError):          # group of 3 is not supported
        m.paged_decode_attention(q2, kc, kc, t, c, 0.1, torch.empty_like(q2))
    kc12 = torch.zeros(4, 4, 12, 128, dtype=torch.bfloat16, device="cuda")
    q4 = torch.zeros(2, 4, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.PkvError):          # block size 12 is not one of 8, 16, 32
        m.paged_decode_attention(q4, kc12, kc12, t, c, 0.1, torch.empty_like(q4))


# ---- the decode step with the cache write folded into the attention launch ----

def run_step(b: BT.Batch, num_warps=0):
    tables, ctx, _ = b.device_index("cuda")
    out = torch.full_like(b.q, float("nan"))
    pkv().paged_decode_step(b.q, b.k_new, b.v_new, b.kc, b.vc, tables, ctx, b.w.scale, out,
                            num_warps=num_warps)
    torch.cuda.synchronize()
    return out


def clone_caches(b: BT.Batch) -> BT.Batch:
    import dataclasses
    return dataclasses.replace(b, kc=b.kc.clone(), vc=b.vc.clone())


@pytest.mark.parametrize("name", list(REDUCED))
@pytest.mark.parametrize("num_warps", [0, 3, 61])
def test_decode_step_equals_write_then_attend(name, num_warps):
    """Fused step: same output bits and same cache bits as the two launches."""
    w, lens = REDUCED[name]
    b = BT.decode_batch(w, lens)
    b2 = clone_caches(b)
    fused = run_step(b, num_warps)
    separate = run(b2, num_warps)
    assert torch.equal(fused, separate)
    assert torch.equal(b.kc.view(torch.int16 if b.kc.element_size() == 2 else torch.int32),
                       b2.kc.view(torch.int16 if b2.kc.element_size() == 2 else torch.int32))
    assert torch.equal(b.vc.view(torch.int16 if b.vc.element_size() == 2 else torch.int32),
                       b2.vc.view(torch.int16 if b2.vc.element_size() == 2 else torch.int32))


@pytest.mark.parametrize("dtype,D,G", [("bf16", 128, 8), ("f16", 64, 1), ("f32", 64, 2),
                                       ("bf16", 256, 4)])
def test_decode_step_edge_lengths_against_oracle(dtype, D, G):
    import dataclasses
    w = dataclasses.replace(W.WORKLOADS["tiny"], dtype=dtype, head_dim=D, num_kv_heads=3,
                            num_q_heads=3 * G, fixed_pool_blocks=0, seed=23)
    lens = np.array([0, 1, 15, 16, 17, 31, 32, 33, 0, 160, 2])
    b = BT.decode_batch(w, lens)
    seqs = list(range(len(lens)))
    ref = BT.oracle_rows(b, seqs)
    got = run_step(b, 2)
    check_rows(b, seqs, got, ref)
    assert torch.all(got[torch.from_numpy(lens == 0).cuda()] == 0)


def test_decode_step_invalid_device_data_matches_write_then_attend():
    """A length past the table, a negative length and a block id outside the pool in
    the last block of a sequence: the fused step writes nothing for those sequences
    (as the cache write with their slots skipped), flags the status word, and its
    output and caches equal the write followed by the attention, bit for bit."""
    m = pkv()
    w, lens = REDUCED["gqa70b"]
    b = BT.decode_batch(w, lens)
    b2 = clone_caches(b)
    tables, ctx, _ = b.device_index("cuda")
    B, MAXB, NB = w.block_size, tables.shape[1], b.kc.shape[0]
    bad_ctx, bad_tab = ctx.clone(), tables.clone()
    bad_ctx[2] = MAXB * B + 5                       # longer than the table can hold
    bad_ctx[3] = -4
    last = (int(bad_ctx[0]) - 1) // B
    bad_tab[0, last] = NB + 1000                    # outside the pool
    # the write of the separate path: the same new tokens, invalid ones skipped
    slots = np.full(len(lens), -1, dtype=np.int32)
    tab_h, ctx_h = bad_tab.cpu().numpy(), bad_ctx.cpu().numpy()
    for s_, t in enumerate(ctx_h):
        if 0 < t <= MAXB * B:
            blk = int(tab_h[s_, (t - 1) // B])
            if 0 <= blk < NB:
                slots[s_] = blk * B + (t - 1) % B
    ws = torch.zeros(m.workspace_bytes(w.num_q_heads, w.num_kv_heads, w.head_dim, b.q.dtype),
                     dtype=torch.uint8, device="cuda")
    ws2 = torch.zeros_like(ws)
    out = torch.full_like(b.q, float("nan"))
    m.paged_decode_step(b.q, b.k_new, b.v_new, b.kc, b.vc, bad_tab, bad_ctx, w.scale, out, ws)
    m.paged_kv_write(b2.k_new, b2.v_new, torch.from_numpy(slots).cuda(), b2.kc, b2.vc)
    out2 = torch.full_like(b.q, float("nan"))
    m.paged_decode_attention(b2.q, b2.kc, b2.vc, bad_tab, bad_ctx, w.scale, out2, ws2)
    torch.cuda.synchronize()
    assert m.decode_status(ws) == m.decode_status(ws2) == 3
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(b.kc.view(torch.int16), b2.kc.view(torch.int16))
    assert torch.equal(b.vc.view(torch.int16), b2.vc.view(torch.int16))


def test_decode_step_full_mha13b_every_row():
    b = BT.decode_batch(W.WORKLOADS["mha13b"])
    seqs = list(range(len(b.lens)))
    ref = BT.oracle_rows(b, seqs)
    check_rows(b, seqs, run_step(b), ref)


@pytest.mark.parametrize("num_warps", [0, 61])
def test_maximum_sequence_count(num_warps):
    """2048 sequences, the most one launch takes, with ragged lengths (1..300, zero
    included): sampled rows against the oracle; one more sequence is refused."""
    import dataclasses
    r = np.random.default_rng(7)
    lens = r.integers(0, 301, 2048)
    lens[:3] = (0, 1, 300)
    w = dataclasses.replace(W.WORKLOADS["gqa70b"], num_q_heads=16, num_kv_heads=2)
    b = BT.decode_batch(w, lens)
    seqs = sorted({0, 1, 2, 2047} | set(r.choice(2048, 12, replace=False).tolist()))
    ref = BT.oracle_rows(b, seqs)
    out = run(b, num_warps)
    check_rows(b, seqs, out, ref)
    assert torch.count_nonzero(out[0]) == 0  # empty context: zero row
    m = pkv()
    q = torch.zeros(2049, 16, 128, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(2049, 1, dtype=torch.int32, device="cuda")
    c = torch.ones(2049, dtype=torch.int32, device="cuda")
    with pytest.raises(m.PkvError):
        m.paged_decode_attention(q, b.kc, b.vc, t, c, 0.1, torch.empty_like(q))

"""GPU parity of paged (chunked) prefill attention against the fp64 oracle.

Row tolerance as for decode (2e-3 of the oracle row's L2 norm, f16/bf16).
Covered: whole-prompt prefills of lengths 1 to several hundred, chunks of 1 to
65 queries at the end of longer contexts, an empty chunk, every group size
{1, 2, 4, 8}, head_dim 64 and 128, f16 and bf16; NaN in every cache slot no
query may read (block tails past the context, unused blocks); a clean status
word; rows outside the chunks left untouched; keys whose magnitude grows with
their position (scores rising along the sequence by many factors of 2^8, so
the kernel's running reference max moves again and again); cache blocks of 8
and 32 tokens (a 128-key tile read as 16 or 4 blocks; lengths ending inside a
block, on a block boundary and on a tile boundary); an output only 16-byte
aligned (the same bits as an aligned one); and the bench's own workload at full
size (16 prompts of 2048 tokens, 70B shape) on sampled rows.
"""
import numpy as np
import pytest
import torch

import batches as BT
from oracle import prefill as opf
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


def case(dtype, Hq, Hkv, D, lens, chunks, seed=11, ramp=False, B=16):
    NB = int(sum(-(-t // B) for t in lens)) + 7
    mgr = BlockManager(NB, B, W.pool_order(NB, seed))
    sids = [mgr.create() for _ in lens]
    for s, t in zip(sids, lens):
        mgr.append(s, int(t))
    maxb = max(1, max(len(mgr.tables[s]) for s in sids))
    tables, ctx = mgr.export_tables(sids, maxb)
    tdt = W.torch_dtype(dtype)
    kc = torch.empty((NB, Hkv, B, D), dtype=tdt, device="cuda")
    vc = torch.empty_like(kc)
    W.fill_normal_(kc, seed, W.STREAM_K_POOL)
    W.fill_normal_(vc, seed, W.STREAM_V_POOL)
    if ramp:  # K at position p scaled by 1 + p / 32
        f = np.ones((NB, B), dtype=np.float32)
        for s, t in enumerate(lens):
            for p in range(t):
                f[tables[s, p // B], p % B] = 1 + p / 32
        kc.mul_(torch.from_numpy(f).cuda().view(NB, 1, B, 1).to(tdt))
    # NaN in every slot no query may read
    used = np.zeros((NB, B), dtype=bool)
    for s, t in enumerate(lens):
        for p in range(t):
            used[tables[s, p // B], p % B] = True
    m = torch.from_numpy(~used).cuda().view(NB, 1, B, 1).expand_as(kc)
    kc[m] = float("nan")
    vc[m] = float("nan")
    qstart = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = W.normal_tensor((int(qstart[-1]) + 3, Hq, D), dtype, seed, W.STREAM_Q, "cuda")
    return kc, vc, q, tables, ctx, qstart


CASES = [
    ("f16", 8, 8, 128, (1, 15, 16, 17, 100, 333), None),
    ("bf16", 64, 8, 128, (40, 700, 129), (40, 65, 1)),
    ("bf16", 16, 4, 64, (33, 64, 500, 31), (7, 64, 0, 31)),
    ("f16", 8, 4, 128, (1000, 17), (200, 17)),
    ("bf16", 8, 1, 128, (300, 96), (300, 33)),
]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,lens,chunks", CASES)
def test_prefill_matches_oracle(dtype, Hq, Hkv, D, lens, chunks):
    chunks = lens if chunks is None else chunks
    kc, vc, q, tables, ctx, qstart = case(dtype, Hq, Hkv, D, lens, chunks)
    T = int(qstart[-1])
    ref = opf.paged_prefill_attention(BT.np64(q[:T]), BT.np64(kc), BT.np64(vc), tables, ctx,
                                      qstart, 1 / np.sqrt(D))
    out = torch.full_like(q, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv().paged_prefill_attention(q, kc, vc, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(ctx).cuda(), torch.from_numpy(qstart).cuda(),
                                  1 / np.sqrt(D), out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = BT.np64(out)
    assert np.all(got[T:] == 7.0)                        # rows past the chunks untouched
    err = BT.row_errors(got[:T], ref)
    assert np.isfinite(got[:T]).all()
    assert err.max() <= BT.tolerance(dtype), f"row error {err.max():.3e}"


@pytest.mark.parametrize("dtype,Hq,Hkv,D,lens,chunks", [
    ("f16", 8, 8, 128, (300, 17), None),
    ("bf16", 16, 4, 64, (200, 129), (200, 50)),
])
def test_prefill_output_only_16_byte_aligned(dtype, Hq, Hkv, D, lens, chunks):
    """The output rows are written 32 bytes at a time when the output allows it; an
    output that is 16-byte aligned but not 32 gets the same bits through 16-byte
    stores, and nothing outside its rows is written."""
    chunks = lens if chunks is None else chunks
    kc, vc, q, tables, ctx, qstart = case(dtype, Hq, Hkv, D, lens, chunks, seed=21)
    args = (torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(),
            torch.from_numpy(qstart).cuda(), 1 / np.sqrt(D))
    out = torch.full_like(q, 7.0)
    pkv().paged_prefill_attention(q, kc, vc, *args, out)
    n = q.numel()
    buf = torch.full((n + 32,), 5.0, dtype=q.dtype, device="cuda")
    shifted = buf[8:8 + n].view(q.shape)      # 16 bytes past a 256-byte aligned start
    assert shifted.data_ptr() % 32 == 16
    shifted.fill_(7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv().paged_prefill_attention(q, kc, vc, *args, shifted, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(shifted.view(torch.int16), out.view(torch.int16))
    assert torch.all(buf[:8] == 5.0) and torch.all(buf[8 + n:] == 5.0)


@pytest.mark.parametrize("dtype,Hq,Hkv,D,lens,chunks", [
    ("bf16", 16, 2, 128, (1000, 300), (1000, 77)),
    ("f16", 8, 8, 64, (700, 129), None),
])
def test_prefill_rising_scores(dtype, Hq, Hkv, D, lens, chunks):
    chunks = lens if chunks is None else chunks
    kc, vc, q, tables, ctx, qstart = case(dtype, Hq, Hkv, D, lens, chunks, seed=13, ramp=True)
    T = int(qstart[-1])
    ref = opf.paged_prefill_attention(BT.np64(q[:T]), BT.np64(kc), BT.np64(vc), tables, ctx,
                                      qstart, 1 / np.sqrt(D))
    out = torch.full_like(q, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv().paged_prefill_attention(q, kc, vc, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(ctx).cuda(), torch.from_numpy(qstart).cuda(),
                                  1 / np.sqrt(D), out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = BT.np64(out)
    assert np.isfinite(got[:T]).all()
    err = BT.row_errors(got[:T], ref)
    assert err.max() <= BT.tolerance(dtype), f"row error {err.max():.3e}"


def test_prefill_last_query_agrees_with_decode_kernel():
    """The last query of each chunk is a decode query at the same context."""
    dtype, Hq, Hkv, D = "bf16", 32, 4, 128
    lens, chunks = (257, 40, 1025), (17, 40, 5)
    kc, vc, q, tables, ctx, qstart = case(dtype, Hq, Hkv, D, lens, chunks, seed=12)
    T = int(qstart[-1])
    out = torch.empty_like(q)
    pkv().paged_prefill_attention(q, kc, vc, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(ctx).cuda(), torch.from_numpy(qstart).cuda(),
                                  0.1, out)
    last = torch.from_numpy(qstart[1:] - 1).long().cuda()
    dec = torch.empty_like(q[last])
    pkv().paged_decode_attention(q[last].contiguous(), kc, vc, torch.from_numpy(tables).cuda(),
                                 torch.from_numpy(ctx).cuda(), 0.1, dec)
    torch.cuda.synchronize()
    ref = BT.np64(dec)
    err = BT.row_errors(BT.np64(out[last]), ref)
    assert err.max() <= 2 * BT.tolerance(dtype)


def test_prefill_bench_size_sampled_rows():
    """The bench's own prefill (70B shape: 16 prompts of 2048 tokens, 64 q / 8 KV heads,
    bf16, whole prompts, one launch over all of them) checked on sampled query rows:
    prefill row p of a prompt equals decode attention at context p + 1, which the
    fp64 oracle computes row by row."""
    from oracle import paged_attention as opa
    from paged_kv_cache_166_gb300 import BlockAllocator
    w = W.WORKLOADS["gqa70b"]
    S, P, B, Hq, Hkv, D = 16, 2048, w.block_size, w.num_q_heads, w.num_kv_heads, w.head_dim
    NB = S * (P // B) + 1
    alloc = BlockAllocator(NB, B, W.pool_order(NB, w.seed))
    sids = [alloc.create() for _ in range(S)]
    for s_ in sids:
        alloc.append(s_, P)
    tables, ctx = alloc.export_tables(sids, P // B)
    kc = torch.empty((NB, Hkv, B, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    W.fill_normal_(kc, w.seed, W.STREAM_K_POOL)
    W.fill_normal_(vc, w.seed, W.STREAM_V_POOL)
    q = W.normal_tensor((S * P, Hq, D), "bf16", w.seed, W.STREAM_Q, "cuda")
    out = torch.empty_like(q)
    qstart = torch.arange(0, S * P + 1, P, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv().paged_prefill_attention(q, kc, vc, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(ctx).cuda(), qstart, w.scale, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(5)
    picks = [(0, 0), (0, 1), (1, 15), (2, 16), (3, 127), (4, 128), (5, 255), (6, 256),
             (15, 2047), (14, 2046)] + [(int(s), int(i)) for s, i in
                                        zip(rng.integers(0, S, 22), rng.integers(0, P, 22))]
    for s, i in picks:
        nb = -(-(i + 1) // B)
        idx = torch.from_numpy(tables[s, :nb].astype(np.int64)).cuda()
        kc_s, vc_s = BT.np64(kc.index_select(0, idx)), BT.np64(vc.index_select(0, idx))
        ref = opa.paged_attention(BT.np64(q[s * P + i])[None], kc_s, vc_s,
                                  np.arange(nb, dtype=np.int32)[None], np.array([i + 1]), w.scale)
        err = BT.row_errors(BT.np64(out[s * P + i])[None], ref)
        assert err.max() <= BT.tolerance("bf16"), f"sequence {s} query {i}: row error {err.max():.3e}"


@pytest.mark.parametrize("seed", range(8))
def test_prefill_random_shapes(seed):
    """Seeded random configurations: group size, head_dim, dtype, number of
    sequences, prompt lengths and chunk lengths (whole prompts, empty chunks and
    chunks of any length) all drawn; every output row against the fp64 oracle."""
    rng = np.random.default_rng(1000 + seed)
    dtype = ["f16", "bf16"][int(rng.integers(0, 2))]
    D = [64, 128][int(rng.integers(0, 2))]
    G = [1, 2, 4, 8][int(rng.integers(0, 4))]
    Hkv = int(rng.integers(1, 3))
    S = int(rng.integers(1, 6))
    lens = tuple(int(x) for x in rng.integers(1, 400, S))
    chunks = tuple(t if rng.random() < 0.4 else int(rng.integers(0, t + 1)) for t in lens)
    kc, vc, q, tables, ctx, qstart = case(dtype, G * Hkv, Hkv, D, lens, chunks, seed=20 + seed)
    T = int(qstart[-1])
    out = torch.full_like(q, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv().paged_prefill_attention(q, kc, vc, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(ctx).cuda(), torch.from_numpy(qstart).cuda(),
                                  1 / np.sqrt(D), out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = BT.np64(out)
    assert np.all(got[T:] == 7.0)
    if T == 0:
        return
    ref = opf.paged_prefill_attention(BT.np64(q[:T]), BT.np64(kc), BT.np64(vc), tables, ctx,
                                      qstart, 1 / np.sqrt(D))
    err = BT.row_errors(got[:T], ref)
    assert np.isfinite(got[:T]).all()
    assert err.max() <= BT.tolerance(dtype), f"row error {err.max():.3e} ({dtype}, D {D}, G {G})"


def test_prefill_maximum_sequence_count():
    """2048 sequences, the most one launch takes (whole prompts and chunks of 0..40
    queries, contexts up to 90 tokens): every row against the oracle; one more
    sequence is refused."""
    r = np.random.default_rng(9)
    lens = tuple(int(x) for x in r.integers(1, 91, 2048))
    chunks = tuple(t if r.random() < 0.3 else int(r.integers(0, min(t, 40) + 1)) for t in lens)
    kc, vc, q, tables, ctx, qstart = case("bf16", 4, 2, 128, lens, chunks, seed=31)
    T = int(qstart[-1])
    ref = opf.paged_prefill_attention(BT.np64(q[:T]), BT.np64(kc), BT.np64(vc), tables, ctx,
                                      qstart, 1 / np.sqrt(128))
    out = torch.full_like(q, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv().paged_prefill_attention(q, kc, vc, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(ctx).cuda(), torch.from_numpy(qstart).cuda(),
                                  1 / np.sqrt(128), out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = BT.np64(out)
    assert np.all(got[T:] == 7.0)
    err = BT.row_errors(got[:T], ref)
    assert err.max() <= BT.tolerance("bf16"), f"row error {err.max():.3e}"
    qs2 = torch.zeros(2050, dtype=torch.int32, device="cuda")
    t2 = torch.zeros(2049, 1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv().PkvError):
        pkv().paged_prefill_attention(q, kc, vc, t2, t2[:, 0].contiguous(), qs2, 0.1, out)


BLOCK_CASES = [
    ("f16", 8, 8, 128, (1, 7, 8, 9, 128, 129, 333), None),
    ("bf16", 64, 8, 128, (40, 700, 256), (40, 65, 1)),
    ("bf16", 16, 4, 64, (33, 64, 500, 31), (7, 64, 0, 31)),
    ("f16", 8, 2, 128, (1000, 31, 32, 33), (200, 31, 1, 33)),
]


@pytest.mark.parametrize("B", [8, 32])
@pytest.mark.parametrize("dtype,Hq,Hkv,D,lens,chunks", BLOCK_CASES)
def test_prefill_block_sizes(B, dtype, Hq, Hkv, D, lens, chunks):
    chunks = lens if chunks is None else chunks
    kc, vc, q, tables, ctx, qstart = case(dtype, Hq, Hkv, D, lens, chunks, seed=17 + B, B=B)
    assert kc.shape[2] == B
    T = int(qstart[-1])
    ref = opf.paged_prefill_attention(BT.np64(q[:T]), BT.np64(kc), BT.np64(vc), tables, ctx,
                                      qstart, 1 / np.sqrt(D))
    out = torch.full_like(q, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv().paged_prefill_attention(q, kc, vc, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(ctx).cuda(), torch.from_numpy(qstart).cuda(),
                                  1 / np.sqrt(D), out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = BT.np64(out)
    assert np.all(got[T:] == 7.0)
    assert np.isfinite(got[:T]).all()
    err = BT.row_errors(got[:T], ref)
    assert err.max() <= BT.tolerance(dtype), f"row error {err.max():.3e}"


@pytest.mark.parametrize("B", [4, 64])
def test_prefill_unsupported_block_size_refused(B):
    kc, vc, q, tables, ctx, qstart = case("f16", 8, 8, 64, (40,), (40,), B=B)
    out = torch.zeros_like(q)
    with pytest.raises(pkv().PkvError):
        pkv().paged_prefill_attention(q, kc, vc, torch.from_numpy(tables).cuda(),
                                      torch.from_numpy(ctx).cuda(),
                                      torch.from_numpy(qstart).cuda(), 0.125, out)
    torch.cuda.synchronize()

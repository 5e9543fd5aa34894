"""Pins of the fp64 attention oracle against things other than itself.

* Paged attention equals contiguous attention exactly ("PagedAttention — how
  vLLM stopped wasting 80%...", section "The PagedAttention kernel": no
  approximation; FAQ "Does PagedAttention change the model's outputs?"): the
  oracle, fed a pool built by a reshape of contiguous K/V (not by the slot
  formula), must match torch's scaled_dot_product_attention in fp64 on the
  contiguous tensors, GQA included.
* Special cases with closed forms: one token gives its value row exactly; equal
  keys (or a zero query) give the mean of the values.
* Physical placement does not matter ("Physical blocks can live anywhere in GPU
  memory", section "The core idea"): any relabelling of physical ids gives a
  bit-identical result; so does sharing blocks instead of private copies.
* Planted mistakes (dropped scale, wrong head grouping, off-by-one position)
  in a copy of the oracle fail the pin.
"""
import numpy as np
import pytest
import torch

from oracle import paged_attention as pa


def _contig_case(seed, S, Hq, Hkv, D, lens, B=16):
    r = np.random.default_rng(seed)
    q = r.standard_normal((S, Hq, D))
    Ks = [r.standard_normal((t, Hkv, D)) for t in lens]
    Vs = [r.standard_normal((t, Hkv, D)) for t in lens]
    return q, Ks, Vs


def _paged_pool(seed, Ks, Vs, B, spare=3):
    """Scatter contiguous per-sequence K/V into a shuffled pool by reshaping
    [t_pad, Hkv, D] -> [n_blocks, B, Hkv, D] -> [n_blocks, Hkv, B, D]."""
    r = np.random.default_rng(seed + 7)
    nblk = [-(-K.shape[0] // B) for K in Ks]
    NB = sum(nblk) + spare
    Hkv, D = Ks[0].shape[1:]
    kc = r.standard_normal((NB, Hkv, B, D))  # garbage everywhere else
    vc = r.standard_normal((NB, Hkv, B, D))
    ids = r.permutation(NB)
    tables = np.zeros((len(Ks), max(nblk) + 2), dtype=np.int32)
    pos = 0
    for s, (K, V) in enumerate(zip(Ks, Vs)):
        n = nblk[s]
        phys = ids[pos:pos + n]
        pos += n
        tables[s, :n] = phys
        pad = n * B - K.shape[0]
        Kp = np.concatenate([K, np.full((pad, Hkv, D), np.nan)]).reshape(n, B, Hkv, D)
        Vp = np.concatenate([V, np.full((pad, Hkv, D), np.nan)]).reshape(n, B, Hkv, D)
        kc[phys] = Kp.transpose(0, 2, 1, 3)
        vc[phys] = Vp.transpose(0, 2, 1, 3)
    return kc, vc, tables


def _sdpa(q, Ks, Vs, scale, G):
    out = np.zeros_like(q)
    for s, (K, V) in enumerate(zip(Ks, Vs)):
        qs = torch.from_numpy(q[s]).unsqueeze(1)                         # [Hq, 1, D]
        Kt = torch.from_numpy(K).transpose(0, 1).repeat_interleave(G, 0)  # [Hq, t, D]
        Vt = torch.from_numpy(V).transpose(0, 1).repeat_interleave(G, 0)
        o = torch.nn.functional.scaled_dot_product_attention(qs, Kt, Vt, scale=scale)
        out[s] = o[:, 0, :].numpy()
    return out


@pytest.mark.parametrize("Hq,Hkv,D,B,lens", [
    (4, 4, 64, 16, (1, 17, 40, 100)),
    (8, 2, 32, 16, (5, 16, 33)),
    (8, 1, 16, 4, (3, 4, 9, 1)),
    (16, 2, 64, 8, (70, 1, 8)),
])
def test_matches_sdpa_on_contiguous_data(Hq, Hkv, D, B, lens):
    S = len(lens)
    q, Ks, Vs = _contig_case(11, S, Hq, Hkv, D, lens, B)
    kc, vc, tables = _paged_pool(11, Ks, Vs, B)
    scale = float(np.float32(1 / np.sqrt(D)))
    got = pa.paged_attention(q, kc, vc, tables, np.array(lens), scale)
    ref = _sdpa(q, Ks, Vs, scale, Hq // Hkv)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_single_token_returns_its_value_row():
    q, Ks, Vs = _contig_case(3, 2, 4, 2, 32, (1, 1))
    kc, vc, tables = _paged_pool(3, Ks, Vs, 16)
    got = pa.paged_attention(q, kc, vc, tables, np.array([1, 1]), 0.125)
    for s in range(2):
        for h in range(4):
            assert np.array_equal(got[s, h], Vs[s][0, h // 2])


def test_equal_keys_or_zero_query_give_mean_of_values():
    r = np.random.default_rng(5)
    t, Hkv, D = 37, 2, 16
    K = np.repeat(r.standard_normal((1, Hkv, D)), t, axis=0)
    V = r.standard_normal((t, Hkv, D))
    q = r.standard_normal((1, 2, D))
    kc, vc, tables = _paged_pool(5, [K], [V], 16)
    got = pa.paged_attention(q, kc, vc, tables, np.array([t]), 0.3)
    np.testing.assert_allclose(got[0], V.mean(axis=0), rtol=0, atol=1e-13)
    K2 = r.standard_normal((t, Hkv, D))
    kc2, vc2, tables2 = _paged_pool(6, [K2], [V], 16)
    got0 = pa.paged_attention(np.zeros((1, 2, D)), kc2, vc2, tables2, np.array([t]), 0.3)
    np.testing.assert_allclose(got0[0], V.mean(axis=0), rtol=0, atol=1e-13)


def test_zero_length_gives_zeros():
    q, Ks, Vs = _contig_case(4, 2, 2, 2, 16, (5, 3))
    kc, vc, tables = _paged_pool(4, Ks, Vs, 16)
    got = pa.paged_attention(q, kc, vc, tables, np.array([0, 3]), 0.25)
    assert np.all(got[0] == 0)
    assert np.any(got[1] != 0)


def test_physical_relabelling_is_bit_identical():
    lens = (1, 17, 40, 100)
    q, Ks, Vs = _contig_case(8, 4, 4, 4, 64, lens)
    kc, vc, tables = _paged_pool(8, Ks, Vs, 16)
    base = pa.paged_attention(q, kc, vc, tables, np.array(lens), 0.125)
    perm = np.random.default_rng(9).permutation(kc.shape[0])   # new id of old block b = perm[b]
    kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
    kc2[perm] = kc; vc2[perm] = vc
    got = pa.paged_attention(q, kc2, vc2, perm[tables].astype(np.int32), np.array(lens), 0.125)
    assert np.array_equal(got, base)


def test_shared_blocks_equal_private_copies_bitwise():
    r = np.random.default_rng(10)
    B, Hkv, D = 16, 2, 32
    prefix_blocks = 3
    NB = 40
    kc = r.standard_normal((NB, Hkv, B, D)); vc = r.standard_normal((NB, Hkv, B, D))
    # two sequences sharing blocks 0..2, private tails 3 and 4
    shared = np.array([[0, 1, 2, 3], [0, 1, 2, 4]], dtype=np.int32)
    # private layout: copy the shared blocks to 10..12 for the second sequence
    kc[10:13] = kc[0:3]; vc[10:13] = vc[0:3]
    private = np.array([[0, 1, 2, 3], [10, 11, 12, 4]], dtype=np.int32)
    q = r.standard_normal((2, 4, D))
    ctx = np.array([prefix_blocks * B + 5, prefix_blocks * B + 9])
    a = pa.paged_attention(q, kc, vc, shared, ctx, 0.2)
    b = pa.paged_attention(q, kc, vc, private, ctx, 0.2)
    assert np.array_equal(a, b)


def _mutant_dropped_scale(q, kc, vc, tables, ctx, scale):
    return pa.paged_attention(q, kc, vc, tables, ctx, 1.0)


def _mutant_head_mapping(q, kc, vc, tables, ctx, scale):
    S, Hq, D = q.shape
    Hkv = kc.shape[1]
    out = np.zeros((S, Hq, D))
    for s in range(S):
        t = int(ctx[s])
        for h in range(Hq):
            g = h % Hkv                       # planted: strided instead of contiguous groups
            K = pa.gather_sequence(kc, tables[s], t, g)
            V = pa.gather_sequence(vc, tables[s], t, g)
            sc = np.float64(np.float32(scale)) * (K @ q[s, h])
            w = np.exp(sc - sc.max())
            out[s, h] = w @ V / w.sum()
    return out


def _mutant_off_by_one(q, kc, vc, tables, ctx, scale):
    return pa.paged_attention(q, kc, vc, tables, np.maximum(np.asarray(ctx) - 1, 1), scale)


@pytest.mark.parametrize("mutant", [_mutant_dropped_scale, _mutant_head_mapping, _mutant_off_by_one])
def test_planted_mistakes_fail_the_sdpa_pin(mutant):
    lens = (5, 16, 33)
    q, Ks, Vs = _contig_case(12, 3, 8, 2, 32, lens)
    kc, vc, tables = _paged_pool(12, Ks, Vs, 16)
    scale = float(np.float32(1 / np.sqrt(32)))
    ref = _sdpa(q, Ks, Vs, scale, 4)
    bad = mutant(q, kc, vc, tables, np.array(lens), scale)
    assert not np.allclose(bad, ref, rtol=1e-6, atol=1e-6)


def test_slot_formula_examples():
    # "What is paged attention?", section "How it works": slot(p) = table[p // 16]*16 + p % 16
    row = [7, 3, 11]
    assert pa.slot_of(row, 0, 16) == 7 * 16
    assert pa.slot_of(row, 15, 16) == 7 * 16 + 15
    assert pa.slot_of(row, 16, 16) == 3 * 16        # "Entry 1 maps to the block holding tokens 16-31"
    assert pa.slot_of(row, 39, 16) == 11 * 16 + 7   # token 39 is in logical block 2 (tokens 32-39)

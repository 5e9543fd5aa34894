"""Pins of the paged prefill oracle against things other than itself.

* A whole-prompt prefill (chunk = the whole context) equals torch's causal
  scaled_dot_product_attention in fp64 on the contiguous K/V the test scatters
  into a shuffled pool by reshaping (MHA and GQA, several block sizes).
* A chunk (the last c positions of a longer context) equals SDPA with the
  explicit mask "key position <= query position".
* The chunk's last query equals single-token decode attention (the decode
  oracle) at the same context; the first position of a prompt returns its value
  row exactly; empty chunks leave their rows untouched.
* A planted off-by-one in the causal limit fails the SDPA pin.
"""
import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from oracle import prefill as pf
from test_oracle_attention import _contig_case, _paged_pool


def _sdpa_masked(q, K, V, scale, G, c):
    """q [c, Hq, D] = the last c positions of contiguous K, V [t, Hkv, D]."""
    t = K.shape[0]
    qs = torch.from_numpy(q).transpose(0, 1)                              # [Hq, c, D]
    Kt = torch.from_numpy(K).transpose(0, 1).repeat_interleave(G, 0)       # [Hq, t, D]
    Vt = torch.from_numpy(V).transpose(0, 1).repeat_interleave(G, 0)
    pos = torch.arange(t - c, t)[:, None]
    mask = torch.arange(t)[None, :] <= pos                                 # [c, t]
    o = torch.nn.functional.scaled_dot_product_attention(qs, Kt, Vt, attn_mask=mask, scale=scale)
    return o.transpose(0, 1).numpy()


def _case(seed, Hq, Hkv, D, lens, chunks, B):
    r = np.random.default_rng(seed)
    _, Ks, Vs = _contig_case(seed, len(lens), Hq, Hkv, D, lens, B)
    kc, vc, tables = _paged_pool(seed, Ks, Vs, B)
    qstart = np.concatenate([[0], np.cumsum(chunks)])
    q = r.standard_normal((int(qstart[-1]), Hq, D))
    return q, Ks, Vs, kc, vc, tables, qstart


@pytest.mark.parametrize("Hq,Hkv,D,B,lens", [
    (4, 4, 32, 16, (1, 17, 40)),
    (8, 2, 16, 4, (9, 33)),
    (8, 1, 16, 8, (23, 5, 64)),
    (4, 2, 16, 32, (31, 32, 33, 70)),
])
def test_whole_prompt_matches_causal_sdpa(Hq, Hkv, D, B, lens):
    q, Ks, Vs, kc, vc, tables, qstart = _case(3, Hq, Hkv, D, lens, lens, B)
    scale = float(np.float32(1 / np.sqrt(D)))
    got = pf.paged_prefill_attention(q, kc, vc, tables, np.array(lens), qstart, scale)
    for s, t in enumerate(lens):
        qs = torch.from_numpy(q[qstart[s]:qstart[s + 1]]).transpose(0, 1)
        Kt = torch.from_numpy(Ks[s]).transpose(0, 1).repeat_interleave(Hq // Hkv, 0)
        Vt = torch.from_numpy(Vs[s]).transpose(0, 1).repeat_interleave(Hq // Hkv, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(qs, Kt, Vt, is_causal=True,
                                                               scale=scale)
        assert np.allclose(got[qstart[s]:qstart[s + 1]], ref.transpose(0, 1).numpy(),
                           rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv,D,B,lens,chunks", [
    (4, 2, 32, 16, (40, 100), (7, 33)),
    (8, 8, 16, 4, (9, 31, 64), (1, 31, 16)),
    (8, 4, 16, 8, (17, 48), (9, 1)),
    (4, 4, 16, 32, (65, 96), (33, 64)),
])
def test_chunk_matches_masked_sdpa(Hq, Hkv, D, B, lens, chunks):
    q, Ks, Vs, kc, vc, tables, qstart = _case(4, Hq, Hkv, D, lens, chunks, B)
    scale = float(np.float32(1 / np.sqrt(D)))
    got = pf.paged_prefill_attention(q, kc, vc, tables, np.array(lens), qstart, scale)
    for s, c in enumerate(chunks):
        ref = _sdpa_masked(q[qstart[s]:qstart[s + 1]], Ks[s], Vs[s], scale, Hq // Hkv, c)
        assert np.allclose(got[qstart[s]:qstart[s + 1]], ref, rtol=1e-12, atol=1e-12)


def test_last_query_equals_decode_and_first_position_is_its_value():
    Hq, Hkv, D, B, lens, chunks = 8, 2, 16, 16, (50, 18, 1), (12, 18, 1)
    q, Ks, Vs, kc, vc, tables, qstart = _case(5, Hq, Hkv, D, lens, chunks, B)
    got = pf.paged_prefill_attention(q, kc, vc, tables, np.array(lens), qstart, 0.25)
    last = q[qstart[1:] - 1]
    dec = pa.paged_attention(last, kc, vc, tables, np.array(lens), 0.25)
    assert np.allclose(got[qstart[1:] - 1], dec, rtol=1e-13, atol=1e-13)
    # sequence 1 is a whole prompt: its first query sees only position 0
    for h in range(Hq):
        assert np.allclose(got[qstart[1], h], Vs[1][0, h // (Hq // Hkv)], rtol=0, atol=1e-15)
    # sequence 2 (one token) too
    assert np.allclose(got[qstart[2]], Vs[2][0].repeat(Hq // Hkv, 0), atol=1e-15)


def test_empty_chunk_leaves_rows_alone():
    Hq, Hkv, D, B, lens, chunks = 4, 4, 16, 16, (20, 30), (0, 5)
    q, Ks, Vs, kc, vc, tables, qstart = _case(6, Hq, Hkv, D, lens, chunks, B)
    sc = float(np.float32(0.3))  # the oracle takes the scale as fp32
    got = pf.paged_prefill_attention(q, kc, vc, tables, np.array(lens), qstart, sc)
    ref = _sdpa_masked(q[0:5], Ks[1], Vs[1], sc, 1, 5)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_planted_off_by_one_fails_the_pin():
    Hq, Hkv, D, B, lens, chunks = 4, 2, 16, 16, (40,), (9,)
    q, Ks, Vs, kc, vc, tables, qstart = _case(7, Hq, Hkv, D, lens, chunks, B)
    sc = float(np.float32(0.3))
    ref = _sdpa_masked(q, Ks[0], Vs[0], sc, 2, 9)
    # the oracle with "j < p" instead of "j <= p": the same call one position earlier
    wrong = pf.paged_prefill_attention(q, kc, vc, tables, np.array([39]), qstart, sc)
    assert not np.allclose(wrong, ref, rtol=1e-6, atol=1e-6)
    right = pf.paged_prefill_attention(q, kc, vc, tables, np.array([40]), qstart, sc)
    assert np.allclose(right, ref, rtol=1e-12, atol=1e-12)

"""Pins of the fp8 (E4M3) KV-cache oracle against things other than itself.

The pages name a quantised KV cache (K/V in int8 or fp8 instead of fp16) as
orthogonal to paging and composable with it ("PagedAttention — how vLLM
stopped wasting 80% of your GPU memory", FAQ "How does this relate to
quantization?") and fix no format; the oracle reads it as E4M3 codes with one
fp32 scale per KV head, round to nearest even, saturating.

* The code table against the format's closed forms: smallest subnormal 2^-9,
  smallest normal 2^-6, one, largest finite 448, NaN patterns, sign symmetry,
  127 strictly increasing finite magnitudes.
* Encoding against brute force: every finite code round-trips; every midpoint
  of two neighbours goes to the even code and just off it to the nearer one;
  random values land on a nearest representable value; out-of-range values
  saturate to +-448, NaN gives 0x7F.
* Encoding against a library routine: torch's float8_e4m3fn cast on in-range
  values.
* Quantised attention: with K/V that E4M3 represents exactly (times the per-head
  scales), attention over the fp8 pool equals torch's fp64 SDPA on the
  contiguous values; dequantisation error stays within half a code step.
* Layout: a written token lands at [block, head, offset, :] in K and at
  [block, head, :, byte of offset] in V (the byte order is a permutation of
  the 16 tokens); padding slots are skipped.
"""
import numpy as np
import pytest
import torch

from oracle import fp8
from test_oracle_attention import _paged_pool, _sdpa


def test_code_table_closed_forms():
    assert fp8.decode(0x00) == 0.0
    assert fp8.decode(0x01) == 2.0 ** -9
    assert fp8.decode(0x07) == 7 * 2.0 ** -9
    assert fp8.decode(0x08) == 2.0 ** -6
    assert fp8.decode(0x38) == 1.0
    assert fp8.decode(0x39) == 1.125
    assert fp8.decode(0x7E) == 448.0
    assert np.isnan(fp8.decode(0x7F)) and np.isnan(fp8.decode(0xFF))
    codes = np.arange(0x7F)
    mags = fp8.decode(codes)
    assert np.all(np.diff(mags) > 0)
    assert np.array_equal(fp8.decode(codes | 0x80), -mags)


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    assert np.array_equal(fp8.encode(fp8.decode(codes)), codes)


def test_midpoints_round_to_the_even_code():
    mags = fp8.decode(np.arange(0x7F))
    for c in range(0x7E):
        mid = 0.5 * (mags[c] + mags[c + 1])
        even = c if c % 2 == 0 else c + 1
        assert fp8.encode(mid) == even
        assert fp8.encode(-mid) == even | 0x80
        assert fp8.encode(np.nextafter(mid, 0)) == c
        assert fp8.encode(np.nextafter(mid, np.inf)) == c + 1


def test_random_values_land_on_a_nearest_code():
    r = np.random.default_rng(0)
    x = np.concatenate([r.standard_normal(4000) * s for s in (1e-3, 0.1, 1, 30, 300)])
    mags = fp8.decode(np.arange(0x7F))
    got = fp8.decode(fp8.encode(x))
    best = np.min(np.abs(np.abs(x)[:, None] - mags[None, :]), axis=1)
    assert np.array_equal(np.abs(np.abs(x) - np.abs(got)), best)
    assert np.array_equal(np.signbit(got), np.signbit(x))


def test_saturation_and_nan():
    assert list(fp8.encode([448.0, 460.0, 464.0, 1e6, np.inf])) == [0x7E] * 5
    assert list(fp8.encode([-448.0, -1e30, -np.inf])) == [0xFE] * 3
    assert fp8.encode(np.nan) == fp8.NAN_CODE


def test_encode_matches_torch_cast_in_range():
    r = np.random.default_rng(1)
    x = np.concatenate([r.standard_normal(20000) * s for s in (0.01, 1.0, 50.0)])
    x = np.clip(x, -440, 440).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode(x), ref)


def test_quantize_error_within_half_a_step():
    r = np.random.default_rng(2)
    x = r.standard_normal(50000).astype(np.float32) * 3
    scale = np.float32(0.05)
    back = fp8.decode(fp8.quantize(x, scale)) * np.float64(scale)
    a = np.abs(x / np.float64(scale))
    # half a step: 2^-4 relative for normals, 2^-10 absolute among subnormals
    bound = np.where(a >= 2.0 ** -6, a * 2.0 ** -4, 2.0 ** -10) * np.float64(scale)
    assert np.all(np.abs(back - x) <= bound * (1 + 1e-12))


def test_v_byte_order_is_a_permutation():
    assert sorted(fp8.V_TOKEN.tolist()) == list(range(16))
    assert np.array_equal(fp8.V_TOKEN[fp8.V_POS], np.arange(16))


@pytest.mark.parametrize("slot", [0, 9, 18, 31])
def test_write_layout_and_padding(slot):
    NB, Hkv, B, D = 3, 2, 16, 8
    kc = np.zeros((NB, Hkv, B, D), np.uint8)
    vc = np.zeros((NB, Hkv, D, B), np.uint8)
    k = np.full((2, Hkv, D), 1.0, np.float32)
    v = np.full((2, Hkv, D), 2.0, np.float32)
    k[1] = -1.0
    fp8.kv_write_fp8(k, v, [slot, -1], [1.0, 0.5], [1.0, 4.0], kc, vc)
    blk, off = slot // B, slot % B
    assert np.all(kc[blk, 0, off] == 0x38) and np.all(kc[blk, 1, off] == 0x40)  # 1.0, 2.0
    byte = int(fp8.V_POS[off])
    assert np.all(vc[blk, 0, :, byte] == 0x40) and np.all(vc[blk, 1, :, byte] == 0x30)  # 2.0, 0.5
    assert np.count_nonzero(kc) == Hkv * D and np.count_nonzero(vc) == Hkv * D


@pytest.mark.parametrize("Hq,Hkv,D,lens", [(4, 4, 32, (1, 17, 40)), (8, 2, 16, (5, 33))])
def test_attention_on_representable_values_matches_sdpa(Hq, Hkv, D, lens):
    B = 16
    r = np.random.default_rng(3)
    k_scale = np.array([0.25, 0.5, 1.0, 2.0][:Hkv], np.float32)
    v_scale = np.array([1.0, 0.125, 0.5, 4.0][:Hkv], np.float32)
    mags = fp8.decode(np.arange(0x7F))
    # K/V: random exactly representable codes times the head's scale
    Kc = [r.choice(np.concatenate([mags, -mags[1:]]), size=(t, Hkv, D)) for t in lens]
    Vc = [r.choice(np.concatenate([mags, -mags[1:]]), size=(t, Hkv, D)) for t in lens]
    Ks = [K * k_scale.astype(np.float64)[None, :, None] for K in Kc]
    Vs = [V * v_scale.astype(np.float64)[None, :, None] for V in Vc]
    q = r.standard_normal((len(lens), Hq, D)) * 0.05
    kf, vf, tables = _paged_pool(5, Ks, Vs, B)
    kf = np.nan_to_num(kf)
    vf = np.nan_to_num(vf)
    # quantise the pool (the values are exactly representable); V tiles transposed,
    # tokens in the V byte order
    k8 = fp8.quantize(kf, k_scale[None, :, None, None])
    vt = np.swapaxes(fp8.quantize(vf, v_scale[None, :, None, None]), 2, 3)
    v8 = np.ascontiguousarray(vt[..., fp8.V_TOKEN])
    scale = float(np.float32(1 / np.sqrt(D)))
    got = fp8.paged_attention_fp8(q, k8, v8, k_scale, v_scale, tables, np.array(lens), scale)
    ref = _sdpa(q, Ks, Vs, scale, Hq // Hkv)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)

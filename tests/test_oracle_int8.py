"""Pins of the int8 KV-cache oracle against things other than itself.

The pages list int8 next to fp8 as a quantised KV-cache element type
("PagedAttention — how vLLM stopped wasting 80% of your GPU memory", FAQ "How
does this relate to quantization?") and fix no format; the oracle reads it as
symmetric codes in [-127, 127] with one fp32 scale per KV head, the fp32
quotient rounded to the nearest integer with ties to even.

* Hand-worked values: ties go to the even integer (0.5 -> 0, 1.5 -> 2,
  2.5 -> 2, -2.5 -> -2), the range is clamped at +-127 (127.5 and 1e9 -> 127,
  -128 is never written), infinities saturate and NaN gives 0.
* Brute force: the code is the integer in [-127, 127] nearest to the fp32
  quotient (all 255 candidates compared), ties to the even one.
* Library routine: torch's round (half to even) of torch's fp32 division,
  clamped, on random values; and one worked case whose fp32 quotient is a tie
  that the exact quotient is not (30.424475 / 0.54818875 -> 55.5 -> 56, where
  the fp64 quotient would give 55).
* Dequantisation error within half a step (scale / 2) inside the range.
* Layout: a written token lands at [block, head, offset, :] in K and at
  [block, head, :, V_POS[offset]] in V; padding slots are skipped.
* Attention over K/V that int8 represents exactly (integers times the per-head
  scales) equals torch's fp64 SDPA on the contiguous values.
"""
import numpy as np
import pytest
import torch

from oracle import fp8, int8
from test_oracle_attention import _paged_pool, _sdpa


def test_hand_worked_values():
    x = [0.0, 0.49, 0.5, 0.51, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 126.5, 127.49, 127.5,
         128.0, 1e9, -127.5, -128.0, -1e9, np.inf, -np.inf, np.nan]
    want = [0, 0, 0, 1, 2, 2, 0, -2, -2, 4, 126, 127, 127, 127, 127, -127, -127, -127, 127,
            -127, 0]
    assert int8.quantize(x, 1.0).tolist() == want
    # the scale divides: x = 3 * 0.25 -> 3 / 0.25 = 12
    assert int8.quantize([0.75, -0.75, 0.125], 0.0625).tolist() == [12, -12, 2]


@pytest.mark.parametrize("scale", [0.37, 0.25])
def test_nearest_code_by_brute_force(scale):
    r = np.random.default_rng(0)
    x = np.concatenate([r.standard_normal(3000) * s for s in (0.01, 1, 10, 100)])
    x = np.concatenate([x, (np.arange(-130, 131) + 0.5) * scale])  # ties when scale = 1/4
    scale = np.float32(scale)
    q = (x.astype(np.float32) / scale).astype(np.float64)        # the fp32 quotient
    codes = np.arange(-127, 128, dtype=np.float64)
    d = np.abs(q[:, None] - codes[None, :])
    first = codes[np.argmin(d, axis=1)]                          # the lower of two nearest
    tie = (d == d.min(axis=1, keepdims=True)).sum(axis=1) > 1
    pick = np.where(tie & (first % 2 != 0), first + 1, first)
    assert np.array_equal(int8.quantize(x, scale).astype(np.float64), pick)
    if scale == np.float32(0.25):
        assert tie.sum() == 254                                  # -126.5 .. 126.5


def test_matches_torch_round_of_fp32_division():
    r = np.random.default_rng(1)
    x = (r.standard_normal(50000) * 40).astype(np.float32)
    s = np.float32(0.29)
    ref = torch.round(torch.from_numpy(x) / torch.tensor(s)).clamp(-127, 127).to(torch.int8)
    assert np.array_equal(int8.quantize(x, s), ref.numpy())
    # a quotient that is a tie in fp32 but not exactly
    x1, s1 = np.float32(30.424475), np.float32(0.54818875)
    assert (torch.tensor(x1) / torch.tensor(s1)).item() == 55.5
    assert np.float64(x1) / np.float64(s1) < 55.5
    assert int8.quantize(x1, s1) == 56


def test_dequantisation_error_within_half_a_step():
    r = np.random.default_rng(2)
    s = np.float32(0.05)
    x = np.clip(r.standard_normal(50000) * 3, -127 * 0.05, 127 * 0.05).astype(np.float32)
    back = int8.decode(int8.quantize(x, s)) * np.float64(s)
    # half a step plus the fp32 quotient's rounding
    assert np.all(np.abs(back - x) <= np.float64(s) * (0.5 + 2.0 ** -17))
    assert int8.decode(np.array([-127, 0, 127], dtype=np.int8)).tolist() == [-127.0, 0.0, 127.0]


@pytest.mark.parametrize("slot", [0, 9, 18, 31])
def test_write_layout_and_padding(slot):
    NB, Hkv, B, D = 3, 2, 16, 8
    kc = np.zeros((NB, Hkv, B, D), np.int8)
    vc = np.zeros((NB, Hkv, D, B), np.int8)
    k = np.full((2, Hkv, D), 1.0, np.float32)
    v = np.full((2, Hkv, D), 2.0, np.float32)
    k[1] = -1.0
    int8.kv_write_int8(k, v, [slot, -1], [0.5, 0.25], [1.0, 0.125], kc, vc)
    blk, off = slot // B, slot % B
    assert np.all(kc[blk, 0, off] == 2) and np.all(kc[blk, 1, off] == 4)
    byte = int(fp8.V_POS[off])
    assert np.all(vc[blk, 0, :, byte] == 2) and np.all(vc[blk, 1, :, byte] == 16)
    assert np.count_nonzero(kc) == Hkv * D and np.count_nonzero(vc) == Hkv * D


@pytest.mark.parametrize("Hq,Hkv,D,lens", [(4, 4, 32, (1, 17, 40)), (8, 2, 16, (5, 33))])
def test_attention_on_representable_values_matches_sdpa(Hq, Hkv, D, lens):
    B = 16
    r = np.random.default_rng(3)
    k_scale = np.array([0.01, 0.02, 0.005, 0.04][:Hkv], np.float32)
    v_scale = np.array([0.03, 0.0125, 0.02, 0.01][:Hkv], np.float32)
    Kc = [r.integers(-127, 128, size=(t, Hkv, D)).astype(np.float64) for t in lens]
    Vc = [r.integers(-127, 128, size=(t, Hkv, D)).astype(np.float64) for t in lens]
    Ks = [K * k_scale.astype(np.float64)[None, :, None] for K in Kc]
    Vs = [V * v_scale.astype(np.float64)[None, :, None] for V in Vc]
    q = r.standard_normal((len(lens), Hq, D))
    kf, vf, tables = _paged_pool(5, Ks, Vs, B)
    kf = np.nan_to_num(kf)
    vf = np.nan_to_num(vf)
    k8 = int8.quantize(kf, k_scale[None, :, None, None])
    vt = np.swapaxes(int8.quantize(vf, v_scale[None, :, None, None]), 2, 3)
    v8 = np.ascontiguousarray(vt[..., fp8.V_TOKEN])
    scale = float(np.float32(1 / np.sqrt(D)))
    got = int8.paged_attention_int8(q, k8, v8, k_scale, v_scale, tables, np.array(lens), scale)
    ref = _sdpa(q, Ks, Vs, scale, Hq // Hkv)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)

"""GPU parity of the fp8 (E4M3) KV cache against the fp64 oracle.

* The quantising cache write is bit-exact against the oracle's (codes compared
  as bytes), for f32/f16/bf16 inputs spanning subnormal, normal and saturating
  magnitudes, with padding slots, out-of-pool slots and every slot of a block.
* Decode attention over fp8 caches matches the oracle's fp64 attention over the
  dequantised codes within the row tolerance of the 16-bit path (2e-3 of the
  row's L2 norm), on reduced versions of the workload shapes under several
  warp counts, on edge lengths with NaN codes in every unused slot and block,
  for head_dim 128 and 256 and all group sizes, and on sampled rows of the
  full-size 13B, 70B and long-context batches in the launch configuration
  bench.py times.
* The fp8 decode step equals the quantising write followed by the attention,
  bit for bit (output and caches), and results are bit-identical between runs.
"""
import numpy as np
import pytest
import torch

import batches as BT
from oracle import fp8 as ofp8
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


class Fp8Batch:
    """A decode batch (tables, lengths, new tokens, q from BT.decode_batch) with
    fp8 caches of seeded codes and per-head scales."""

    def __init__(self, w, lens, canaries=False, **kw):
        b = BT.decode_batch(w, lens, **kw)
        self.b = b
        NB, Hkv, D = b.NB, w.num_kv_heads, w.head_dim
        self.k_scale_h = W.fp8_scales(Hkv, w.seed)
        self.v_scale_h = W.fp8_scales(Hkv, w.seed + 1)
        self.k_scale = torch.from_numpy(self.k_scale_h).cuda()
        self.v_scale = torch.from_numpy(self.v_scale_h).cuda()
        self.kc = torch.empty((NB, Hkv, 16, D), dtype=torch.uint8, device="cuda")
        self.vc = torch.empty((NB, Hkv, D, 16), dtype=torch.uint8, device="cuda")
        W.fill_fp8_codes_(self.kc, self.k_scale_h, w.seed, W.STREAM_K_POOL)
        W.fill_fp8_codes_(self.vc, self.v_scale_h, w.seed, W.STREAM_V_POOL)
        if canaries:
            self._plant_nan_codes()
        # the oracle's copies, taken before any library kernel touches the caches
        self.kc_host = self.kc.cpu().numpy()
        self.vc_host = self.vc.cpu().numpy()

    def _plant_nan_codes(self):
        """NaN codes in every slot no sequence reaches (tails of last blocks, unused
        blocks); the new tokens' slots are overwritten by the write."""
        b = self.b
        used = np.zeros((b.NB, 16), dtype=bool)
        for s in range(len(b.lens)):
            t = int(b.ctx[s])
            for p in range(t):
                used[b.tables[s, p // 16], p % 16] = True
        mask = torch.from_numpy(~used).cuda()
        self.kc[mask.view(b.NB, 1, 16, 1).expand_as(self.kc)] = 0x7F
        # byte j of a V row holds token V_TOKEN[j]
        vtok = torch.from_numpy(ofp8.V_TOKEN).cuda()
        vmask = mask[:, vtok].reshape(b.NB, 1, 1, 16).expand_as(self.vc)
        self.vc[vmask] = 0xFF

    def write(self):
        tables, ctx, slots = self.b.device_index("cuda")
        pkv().paged_kv_write_fp8(self.b.k_new, self.b.v_new, slots, self.kc, self.vc,
                                 self.k_scale, self.v_scale)

    def attend(self, num_warps=0):
        tables, ctx, _ = self.b.device_index("cuda")
        out = torch.full_like(self.b.q, float("nan"))
        pkv().paged_decode_attention_fp8(self.b.q, self.kc, self.vc, self.k_scale, self.v_scale,
                                         tables, ctx, self.b.w.scale, out, num_warps=num_warps)
        torch.cuda.synchronize()
        return out

    def oracle_rows(self, seqs):
        """fp64 oracle rows: the oracle's own quantising write of the new tokens into
        its copy of the codes, then attention over the dequantised codes."""
        b = self.b
        kc, vc = self.kc_host.copy(), self.vc_host.copy()
        sel = torch.tensor(seqs, dtype=torch.long, device="cuda")
        slots = b.new_slots[seqs]
        ofp8.kv_write_fp8(BT.np64(b.k_new.index_select(0, sel)).astype(np.float32),
                          BT.np64(b.v_new.index_select(0, sel)).astype(np.float32),
                          slots, self.k_scale_h, self.v_scale_h, kc, vc)
        return ofp8.paged_attention_fp8(BT.np64(b.q.index_select(0, sel)), kc, vc,
                                        self.k_scale_h, self.v_scale_h, b.tables[seqs],
                                        b.ctx[seqs], b.w.scale)


def check(fb, seqs, got, ref):
    err = BT.row_errors(BT.np64(got)[seqs], ref)
    tol = BT.tolerance(fb.b.w.dtype)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, f"row error {err.max():.3e} > {tol} at {worst}"


def fp8_workload(name, **kw):
    import dataclasses
    w = W.WORKLOADS[name]
    if w.dtype == "f32":
        kw.setdefault("dtype", "f16")
    return dataclasses.replace(w, **kw)


# ---- quantising write ---------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_fp8_write_bit_exact(dtype):
    r = np.random.default_rng(7)
    NB, Hkv, D, T = 6, 3, 128, 70
    k_scale = np.array([0.01, 0.5, 2.0], np.float32)
    v_scale = np.array([0.25, 0.003, 1.0], np.float32)
    # magnitudes from subnormal to beyond the range (saturation)
    mag = np.exp(r.uniform(np.log(1e-4), np.log(2e3), (T, Hkv, D)))
    k = (mag * r.choice([-1, 1], mag.shape)).astype(np.float32)
    v = (np.roll(mag, 1, axis=2) * r.choice([-1, 1], mag.shape)).astype(np.float32)
    tdt = W.torch_dtype(dtype)
    kt, vt = torch.from_numpy(k).to(tdt).cuda(), torch.from_numpy(v).to(tdt).cuda()
    slots = r.permutation(NB * 16)[:T].astype(np.int32)
    slots[::11] = -1                      # padding
    slots[5] = NB * 16 + 3                # past the pool: skipped
    kc = torch.zeros((NB, Hkv, 16, D), dtype=torch.uint8, device="cuda")
    vc = torch.zeros((NB, Hkv, D, 16), dtype=torch.uint8, device="cuda")
    pkv().paged_kv_write_fp8(kt, vt, torch.from_numpy(slots).cuda(), kc, vc,
                             torch.from_numpy(k_scale).cuda(), torch.from_numpy(v_scale).cuda())
    torch.cuda.synchronize()
    okc = np.zeros((NB, Hkv, 16, D), np.uint8)
    ovc = np.zeros((NB, Hkv, D, 16), np.uint8)
    o_slots = np.where(slots < NB * 16, slots, -1)
    ofp8.kv_write_fp8(BT.np64(kt).astype(np.float32), BT.np64(vt).astype(np.float32), o_slots,
                      k_scale, v_scale, okc, ovc)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)


# ---- attention ----------------------------------------------------------------------

REDUCED = [
    ("mha13b", dict(num_q_heads=8, num_kv_heads=8), (300, 1, 2048, 77, 16, 513, 129, 31, 0, 45)),
    ("gqa70b", dict(num_q_heads=32, num_kv_heads=4), (1024, 5, 3000, 16, 17, 700, 1, 2100)),
    ("prefix", dict(), (1000, 1200, 1017, 1512, 3)),
    ("longctx", dict(num_q_heads=16, num_kv_heads=2), (9000, 6000)),
]


@pytest.mark.parametrize("name,kw,lens", REDUCED)
@pytest.mark.parametrize("num_warps", [0, 3, 61])
def test_fp8_attention_matches_oracle(name, kw, lens, num_warps):
    fb = Fp8Batch(fp8_workload(name, **kw), np.asarray(lens))
    seqs = list(range(len(lens)))
    ref = fb.oracle_rows(seqs)
    fb.write()
    check(fb, seqs, fb.attend(num_warps), ref)


@pytest.mark.parametrize("dtype,D,G", [("f16", 128, 1), ("bf16", 128, 8), ("bf16", 256, 2),
                                       ("f16", 256, 4), ("bf16", 128, 4)])
def test_fp8_edge_lengths_with_nan_codes(dtype, D, G):
    lens = np.array([0, 1, 15, 16, 17, 31, 32, 33, 64 * 16])
    w = fp8_workload("gqa70b", dtype=dtype, head_dim=D, num_kv_heads=2, num_q_heads=2 * G)
    fb = Fp8Batch(w, lens, canaries=True, maxb_extra=0)
    seqs = list(range(len(lens)))
    ref = fb.oracle_rows(seqs)
    fb.write()
    out = fb.attend()
    assert torch.isfinite(out).all()
    check(fb, seqs, out, ref)
    assert torch.count_nonzero(out[0]) == 0  # empty context: zero row


def test_fp8_step_equals_write_then_attend_and_is_deterministic():
    w = fp8_workload("gqa70b", num_q_heads=16, num_kv_heads=2)
    lens = np.array([700, 1, 33, 2048, 16, 900])
    a = Fp8Batch(w, lens)
    b = Fp8Batch(w, lens)
    a.write()
    out_a = a.attend()
    out_a2 = a.attend()
    tables, ctx, _ = b.b.device_index("cuda")
    out_b = torch.full_like(b.b.q, float("nan"))
    pkv().paged_decode_step_fp8(b.b.q, b.b.k_new, b.b.v_new, b.kc, b.vc, b.k_scale, b.v_scale,
                                tables, ctx, w.scale, out_b)
    torch.cuda.synchronize()
    assert torch.equal(a.kc, b.kc) and torch.equal(a.vc, b.vc)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(out_a.view(torch.int16), out_a2.view(torch.int16))
    ref = b.oracle_rows(list(range(len(lens))))
    check(b, list(range(len(lens))), out_b, ref)


@pytest.mark.parametrize("name", ["mha13b", "gqa70b", "longctx"])
def test_fp8_full_batches_sampled_rows(name):
    """The bench's full-size batches (13B, 70B and long-context shapes) in the launch
    configuration the bench times, on sampled rows: the shortest and longest
    sequences and random ones (fewer on the long-context batch, whose sequences run
    to 131k tokens)."""
    fb = Fp8Batch(fp8_workload(name), None)
    lens = fb.b.lens
    order = np.argsort(lens)
    r = np.random.default_rng(0)
    if name == "longctx":
        seqs = sorted({int(order[0]), int(order[len(lens) // 2])})
    else:
        seqs = sorted(set([int(order[0]), int(order[-1]), int(order[-2])] +
                          r.choice(len(lens), 5, replace=False).tolist()))
    ref = fb.oracle_rows(seqs)
    fb.write()
    check(fb, seqs, fb.attend(), ref)


def test_fp8_rejections():
    from paged_kv_cache_166_gb300 import _native as N
    fb = Fp8Batch(fp8_workload("gqa70b", num_q_heads=16, num_kv_heads=2), np.array([40, 3]))
    tables, ctx, _ = fb.b.device_index("cuda")
    out = torch.zeros_like(fb.b.q)
    with pytest.raises(ValueError):  # wrong scale shape
        pkv().paged_decode_attention_fp8(fb.b.q, fb.kc, fb.vc, fb.k_scale[:1], fb.v_scale,
                                         tables, ctx, 0.1, out)
    with pytest.raises(ValueError):  # V cache not transposed
        pkv().paged_decode_attention_fp8(fb.b.q, fb.kc, fb.kc, fb.k_scale, fb.v_scale,
                                         tables, ctx, 0.1, out)
    q32 = fb.b.q.float()
    with pytest.raises(N.PkvError):  # f32 q is not supported over fp8 caches
        pkv().paged_decode_attention_fp8(q32, fb.kc, fb.vc, fb.k_scale, fb.v_scale,
                                         tables, ctx, 0.1, torch.zeros_like(q32))
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0

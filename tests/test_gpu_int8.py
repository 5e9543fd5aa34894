"""GPU parity of the int8 KV cache against the fp64 oracle.

* The quantising cache write is bit-exact against the oracle's (codes compared
  as bytes), for f32/f16/bf16 inputs spanning tiny, in-range and saturating
  magnitudes, exact ties, infinities and NaN, with padding and out-of-pool slots.
* Decode attention over int8 caches matches the oracle's fp64 attention over
  the dequantised codes within the row tolerance of the 16-bit path (2e-3 of the
  row's L2 norm): reduced versions of the workload shapes under several warp
  counts; every byte value (-128 included) read back exactly; edge lengths with
  extreme codes in every unused slot and block; head_dim 128 and 256 and all
  group sizes; sampled rows of the full-size 13B, 70B and long-context batches
  in the launch configuration bench.py times.
* The int8 decode step equals the quantising write followed by the attention,
  bit for bit (output and caches), and results are bit-identical between runs.
"""
import dataclasses

import numpy as np
import pytest
import torch

import batches as BT
from oracle import fp8 as ofp8
from oracle import int8 as oi8
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


class Int8Batch:
    """A decode batch (tables, lengths, new tokens, q from BT.decode_batch) with
    int8 caches of seeded codes and per-head scales."""

    def __init__(self, w, lens, canaries=False, all_bytes=False, **kw):
        b = BT.decode_batch(w, lens, **kw)
        self.b = b
        NB, Hkv, D = b.NB, w.num_kv_heads, w.head_dim
        self.k_scale_h = W.int8_scales(Hkv, w.seed)
        self.v_scale_h = W.int8_scales(Hkv, w.seed + 1)
        self.k_scale = torch.from_numpy(self.k_scale_h).cuda()
        self.v_scale = torch.from_numpy(self.v_scale_h).cuda()
        self.kc = torch.empty((NB, Hkv, 16, D), dtype=torch.int8, device="cuda")
        self.vc = torch.empty((NB, Hkv, D, 16), dtype=torch.int8, device="cuda")
        if all_bytes:
            # every byte value, -128 included (never written, but read exactly)
            g = torch.Generator(device="cuda")
            g.manual_seed(w.seed)
            self.kc.copy_(torch.randint(-128, 128, self.kc.shape, generator=g, device="cuda"))
            self.vc.copy_(torch.randint(-128, 128, self.vc.shape, generator=g, device="cuda"))
        else:
            W.fill_int8_codes_(self.kc, self.k_scale_h, w.seed, W.STREAM_K_POOL)
            W.fill_int8_codes_(self.vc, self.v_scale_h, w.seed, W.STREAM_V_POOL)
        if canaries:
            self._plant_extreme_codes()
        self.kc_host = self.kc.cpu().numpy()
        self.vc_host = self.vc.cpu().numpy()

    def _plant_extreme_codes(self):
        """Code 127 in K and -128 in V in every slot no sequence reaches (tails of
        last blocks, unused blocks): read as context, they would dominate the
        scores; the new tokens' slots are overwritten by the write."""
        b = self.b
        used = np.zeros((b.NB, 16), dtype=bool)
        for s in range(len(b.lens)):
            for p in range(int(b.ctx[s])):
                used[b.tables[s, p // 16], p % 16] = True
        mask = torch.from_numpy(~used).cuda()
        self.kc[mask.view(b.NB, 1, 16, 1).expand_as(self.kc)] = 127
        vtok = torch.from_numpy(ofp8.V_TOKEN).cuda()
        vmask = mask[:, vtok].reshape(b.NB, 1, 1, 16).expand_as(self.vc)
        self.vc[vmask] = -128

    def write(self):
        tables, ctx, slots = self.b.device_index("cuda")
        pkv().paged_kv_write_int8(self.b.k_new, self.b.v_new, slots, self.kc, self.vc,
                                  self.k_scale, self.v_scale)

    def attend(self, num_warps=0):
        tables, ctx, _ = self.b.device_index("cuda")
        out = torch.full_like(self.b.q, float("nan"))
        pkv().paged_decode_attention_int8(self.b.q, self.kc, self.vc, self.k_scale, self.v_scale,
                                          tables, ctx, self.b.w.scale, out, num_warps=num_warps)
        torch.cuda.synchronize()
        return out

    def oracle_rows(self, seqs):
        """fp64 oracle rows: the oracle's quantising write of the new tokens into its
        copy of the codes, then attention over the dequantised codes."""
        b = self.b
        kc, vc = self.kc_host.copy(), self.vc_host.copy()
        sel = torch.tensor(seqs, dtype=torch.long, device="cuda")
        oi8.kv_write_int8(BT.np64(b.k_new.index_select(0, sel)).astype(np.float32),
                          BT.np64(b.v_new.index_select(0, sel)).astype(np.float32),
                          b.new_slots[seqs], self.k_scale_h, self.v_scale_h, kc, vc)
        return oi8.paged_attention_int8(BT.np64(b.q.index_select(0, sel)), kc, vc,
                                        self.k_scale_h, self.v_scale_h, b.tables[seqs],
                                        b.ctx[seqs], b.w.scale)


def check(ib, seqs, got, ref):
    err = BT.row_errors(BT.np64(got)[seqs], ref)
    tol = BT.tolerance(ib.b.w.dtype)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, f"row error {err.max():.3e} > {tol} at {worst}"


def int8_workload(name, **kw):
    w = W.WORKLOADS[name]
    if w.dtype == "f32":
        kw.setdefault("dtype", "f16")
    return dataclasses.replace(w, **kw)


# ---- quantising write ---------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_int8_write_bit_exact(dtype):
    r = np.random.default_rng(7)
    NB, Hkv, D, T = 6, 3, 128, 70
    k_scale = np.array([0.01, 0.5, 2.0], np.float32)
    v_scale = np.array([0.25, 0.003, 1.0], np.float32)
    mag = np.exp(r.uniform(np.log(1e-4), np.log(2e3), (T, Hkv, D)))
    k = (mag * r.choice([-1, 1], mag.shape)).astype(np.float32)
    v = (np.roll(mag, 1, axis=2) * r.choice([-1, 1], mag.shape)).astype(np.float32)
    # exact ties of the quotient (x = (n + 1/2) * scale with scale 0.5 or 2.0), and
    # the special values
    k[1, 1, :64] = (np.arange(-32, 32) + 0.5) * 0.5
    k[2, 2, :64] = (np.arange(-32, 32) + 0.5) * 2.0
    k[3, 0, :4] = [np.inf, -np.inf, np.nan, -0.0]
    v[4, 2, :4] = [np.nan, np.inf, -np.inf, 1e30]
    tdt = W.torch_dtype(dtype)
    kt, vt = torch.from_numpy(k).to(tdt).cuda(), torch.from_numpy(v).to(tdt).cuda()
    slots = r.permutation(NB * 16)[:T].astype(np.int32)
    slots[::11] = -1                      # padding (rows 1-4 keep their slots)
    slots[5] = NB * 16 + 3                # past the pool: skipped
    kc = torch.full((NB, Hkv, 16, D), 5, dtype=torch.int8, device="cuda")
    vc = torch.full((NB, Hkv, D, 16), -5, dtype=torch.int8, device="cuda")
    pkv().paged_kv_write_int8(kt, vt, torch.from_numpy(slots).cuda(), kc, vc,
                              torch.from_numpy(k_scale).cuda(), torch.from_numpy(v_scale).cuda())
    torch.cuda.synchronize()
    okc = np.full((NB, Hkv, 16, D), 5, np.int8)
    ovc = np.full((NB, Hkv, D, 16), -5, np.int8)
    o_slots = np.where(slots < NB * 16, slots, -1)
    oi8.kv_write_int8(BT.np64(kt).astype(np.float32), BT.np64(vt).astype(np.float32), o_slots,
                      k_scale, v_scale, okc, ovc)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)
    assert okc.min() >= -127 and ovc[ovc != -5].min() >= -127


# ---- attention ----------------------------------------------------------------------

REDUCED = [
    ("mha13b", dict(num_q_heads=8, num_kv_heads=8), (300, 1, 2048, 77, 16, 513, 129, 31, 0, 45)),
    ("gqa70b", dict(num_q_heads=32, num_kv_heads=4), (1024, 5, 3000, 16, 17, 700, 1, 2100)),
    ("prefix", dict(), (1000, 1200, 1017, 1512, 3)),
    ("longctx", dict(num_q_heads=16, num_kv_heads=2), (9000, 6000)),
]


@pytest.mark.parametrize("name,kw,lens", REDUCED)
@pytest.mark.parametrize("num_warps", [0, 3, 61])
def test_int8_attention_matches_oracle(name, kw, lens, num_warps):
    ib = Int8Batch(int8_workload(name, **kw), np.asarray(lens))
    seqs = list(range(len(lens)))
    ref = ib.oracle_rows(seqs)
    ib.write()
    check(ib, seqs, ib.attend(num_warps), ref)


@pytest.mark.parametrize("D,G", [(128, 1), (128, 8), (256, 2)])
def test_int8_every_byte_value_reads_back(D, G):
    w = int8_workload("gqa70b", head_dim=D, num_kv_heads=2, num_q_heads=2 * G)
    lens = np.array([1, 16, 17, 300, 1000])
    ib = Int8Batch(w, lens, all_bytes=True)
    assert int(ib.kc.min()) == -128 and int(ib.vc.max()) == 127
    seqs = list(range(len(lens)))
    ref = ib.oracle_rows(seqs)
    ib.write()
    check(ib, seqs, ib.attend(), ref)


@pytest.mark.parametrize("dtype,D,G", [("f16", 128, 1), ("bf16", 128, 8), ("bf16", 256, 2),
                                       ("f16", 256, 4), ("bf16", 128, 4)])
def test_int8_edge_lengths_with_extreme_codes(dtype, D, G):
    lens = np.array([0, 1, 15, 16, 17, 31, 32, 33, 64 * 16])
    w = int8_workload("gqa70b", dtype=dtype, head_dim=D, num_kv_heads=2, num_q_heads=2 * G)
    ib = Int8Batch(w, lens, canaries=True, maxb_extra=0)
    seqs = list(range(len(lens)))
    ref = ib.oracle_rows(seqs)
    ib.write()
    out = ib.attend()
    assert torch.isfinite(out).all()
    check(ib, seqs, out, ref)
    assert torch.count_nonzero(out[0]) == 0


def test_int8_step_equals_write_then_attend_and_is_deterministic():
    w = int8_workload("gqa70b", num_q_heads=16, num_kv_heads=2)
    lens = np.array([700, 1, 33, 2048, 16, 900])
    a = Int8Batch(w, lens)
    b = Int8Batch(w, lens)
    a.write()
    out_a = a.attend()
    out_a2 = a.attend()
    tables, ctx, _ = b.b.device_index("cuda")
    out_b = torch.full_like(b.b.q, float("nan"))
    pkv().paged_decode_step_int8(b.b.q, b.b.k_new, b.b.v_new, b.kc, b.vc, b.k_scale, b.v_scale,
                                 tables, ctx, w.scale, out_b)
    torch.cuda.synchronize()
    assert torch.equal(a.kc, b.kc) and torch.equal(a.vc, b.vc)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(out_a.view(torch.int16), out_a2.view(torch.int16))
    ref = b.oracle_rows(list(range(len(lens))))
    check(b, list(range(len(lens))), out_b, ref)


@pytest.mark.parametrize("name", ["mha13b", "gqa70b", "longctx"])
def test_int8_full_batches_sampled_rows(name):
    """The bench's full-size batches (13B, 70B and long-context shapes) in the launch
    configuration the bench times, on sampled rows: the shortest and longest
    sequences and random ones (fewer on the long-context batch, whose sequences run
    to 131k tokens)."""
    ib = Int8Batch(int8_workload(name), None)
    lens = ib.b.lens
    order = np.argsort(lens)
    r = np.random.default_rng(0)
    if name == "longctx":
        seqs = sorted({int(order[0]), int(order[len(lens) // 2])})
    else:
        seqs = sorted(set([int(order[0]), int(order[-1]), int(order[-2])] +
                          r.choice(len(lens), 5, replace=False).tolist()))
    ref = ib.oracle_rows(seqs)
    ib.write()
    check(ib, seqs, ib.attend(), ref)


def test_int8_rejections():
    from paged_kv_cache_166_gb300 import _native as N
    ib = Int8Batch(int8_workload("gqa70b", num_q_heads=16, num_kv_heads=2), np.array([40, 3]))
    tables, ctx, _ = ib.b.device_index("cuda")
    out = torch.zeros_like(ib.b.q)
    with pytest.raises(TypeError):   # an fp8 (uint8) cache handed to the int8 entry
        pkv().paged_decode_attention_int8(ib.b.q, ib.kc.view(torch.uint8), ib.vc.view(torch.uint8),
                                          ib.k_scale, ib.v_scale, tables, ctx, 0.1, out)
    with pytest.raises(ValueError):  # wrong scale shape
        pkv().paged_decode_attention_int8(ib.b.q, ib.kc, ib.vc, ib.k_scale[:1], ib.v_scale,
                                          tables, ctx, 0.1, out)
    q32 = ib.b.q.float()
    with pytest.raises(N.PkvError):  # f32 q is not supported over 8-bit caches
        pkv().paged_decode_attention_int8(q32, ib.kc, ib.vc, ib.k_scale, ib.v_scale,
                                          tables, ctx, 0.1, torch.zeros_like(q32))
    with pytest.raises(N.PkvError):  # int8 caches are not a dtype of the 16-bit write
        N.check(N.lib().pkv_kv_write(ib.b.k_new.data_ptr(), ib.b.v_new.data_ptr(),
                                     tables.data_ptr(), 1, ib.kc.data_ptr(), ib.vc.data_ptr(),
                                     ib.b.NB, 2, 16, 128, N.PKV_INT8, None))
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0

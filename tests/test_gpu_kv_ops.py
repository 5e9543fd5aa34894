"""GPU parity of the cache write and the copy-on-write block copy (bit-exact).

Both kernels are pure data movement, so the device caches must equal the
oracle's caches bit for bit; slots the call does not address keep their canary
bits (compared as raw integers, so NaN canaries count).
"""
import numpy as np
import pytest
import torch

from batches import decode_batch
from oracle import cache_ops
from paged_kv_cache_166_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()


def bits(t: torch.Tensor) -> np.ndarray:
    it = {4: torch.int32, 2: torch.int16}[t.element_size()]
    return t.contiguous().view(it).cpu().numpy()


@pytest.mark.parametrize("dtype,D,Hkv,B", [
    (torch.float32, 64, 4, 16), (torch.float16, 128, 40, 16), (torch.bfloat16, 128, 8, 16),
    (torch.bfloat16, 256, 2, 16), (torch.float16, 64, 3, 8), (torch.bfloat16, 128, 1, 4),
])
def test_kv_write_bit_exact_with_padding_and_canaries(dtype, D, Hkv, B):
    import paged_kv_cache_166_gb300 as pkv
    g = torch.Generator().manual_seed(D * 7 + Hkv)
    NB, T = 37, 53
    k = torch.randn(T, Hkv, D, generator=g).to(dtype)
    v = torch.randn(T, Hkv, D, generator=g).to(dtype)
    slots = torch.randperm(NB * B, generator=g)[:T].to(torch.int32)
    slots[::7] = -1                      # padding tokens
    slots[5] = NB * B + 3                # outside the pool: skipped
    canary = torch.full((NB, Hkv, B, D), float("nan"), dtype=dtype)
    canary.view(torch.int16 if dtype != torch.float32 else torch.int32)[..., ::3] = 0x3C1
    kc, vc = canary.clone().cuda(), (-canary).clone().cuda()
    kc_h, vc_h = canary.float().numpy().copy(), (-canary).float().numpy().copy()
    pkv.paged_kv_write(k.cuda(), v.cuda(), slots.cuda(), kc, vc)
    torch.cuda.synchronize()
    s = slots.numpy().copy()
    s[s >= NB * B] = -1
    kb_exp, vb_exp = bits(canary), bits(-canary)
    k_bits, v_bits = bits(k), bits(v)
    for i, sl in enumerate(s):
        if sl >= 0:
            kb_exp[sl // B, :, sl % B, :] = k_bits[i]
            vb_exp[sl // B, :, sl % B, :] = v_bits[i]
    assert np.array_equal(bits(kc), kb_exp)
    assert np.array_equal(bits(vc), vb_exp)
    # the oracle's scatter agrees on every written value
    cache_ops.kv_write(k.float().numpy(), v.float().numpy(), s, kc_h, vc_h)
    np.testing.assert_array_equal(kc.float().cpu().numpy(), kc_h)
    np.testing.assert_array_equal(vc.float().cpu().numpy(), vc_h)


def test_kv_write_full_gqa70b_decode_step():
    """256 new tokens (one per sequence) of the 70B-shaped batch into its full pool."""
    import paged_kv_cache_166_gb300 as pkv
    b = decode_batch(W.WORKLOADS["gqa70b"])
    tables, ctx, slots = b.device_index("cuda")
    blocks = sorted({int(x) // 16 for x in b.new_slots})
    idx = torch.tensor(blocks, device="cuda")
    exp_k = b.kc.index_select(0, idx).float().cpu().numpy()
    exp_v = b.vc.index_select(0, idx).float().cpu().numpy()
    pkv.paged_kv_write(b.k_new, b.v_new, slots, b.kc, b.vc)
    torch.cuda.synchronize()
    remap = {blk: i for i, blk in enumerate(blocks)}
    local = np.array([remap[int(x) // 16] * 16 + int(x) % 16 for x in b.new_slots], dtype=np.int32)
    cache_ops.kv_write(b.k_new.float().cpu().numpy(), b.v_new.float().cpu().numpy(), local,
                       exp_k, exp_v)
    assert np.array_equal(b.kc.index_select(0, idx).float().cpu().numpy(), exp_k)
    assert np.array_equal(b.vc.index_select(0, idx).float().cpu().numpy(), exp_v)
    # every other block keeps the generator's values (regenerated from the same seed)
    mask = torch.ones(b.NB, dtype=torch.bool, device="cuda")
    mask[idx] = False
    ref = torch.empty_like(b.kc)
    W.fill_normal_(ref, b.w.seed, W.STREAM_K_POOL)
    assert torch.equal(b.kc[mask], ref[mask])
    W.fill_normal_(ref, b.w.seed, W.STREAM_V_POOL)
    assert torch.equal(b.vc[mask], ref[mask])


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_copy_blocks_bit_exact(dtype):
    import paged_kv_cache_166_gb300 as pkv
    g = torch.Generator().manual_seed(3)
    NB, Hkv, B, D = 20, 8, 16, 128
    kc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    vc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    pairs = np.array([[1, 7], [2, 9], [4, 11], [0, 19], [25, 3], [5, -1]], dtype=np.int32)
    kd, vd = kc.cuda(), vc.cuda()
    pkv.paged_copy_blocks(kd, vd, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    kh, vh = kc.float().numpy().copy(), vc.float().numpy().copy()
    valid = pairs[(pairs >= 0).all(1) & (pairs < NB).all(1)]
    cache_ops.copy_blocks(kh, vh, valid)
    assert np.array_equal(kd.float().cpu().numpy(), kh)
    assert np.array_equal(vd.float().cpu().numpy(), vh)


@pytest.mark.parametrize("dtype,L", [(torch.float16, 1), (torch.bfloat16, 5), (torch.uint8, 3),
                                     (torch.int8, 2), (torch.bfloat16, 128)])
def test_copy_blocks_layers_bit_exact(dtype, L):
    """Every layer's caches equal the oracle's per-layer copies, bit for bit, and
    equal L single-layer calls; pairs out of the pool are skipped in every layer."""
    import paged_kv_cache_166_gb300 as pkv
    g = torch.Generator().manual_seed(5 + L)
    NB, Hkv, B, D = 24, 4, 16, 64
    if dtype in (torch.uint8, torch.int8):
        lo, hi = (0, 256) if dtype == torch.uint8 else (-128, 128)
        make = lambda: torch.randint(lo, hi, (NB, Hkv, B, D), generator=g, dtype=dtype)
    else:
        make = lambda: torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    kh = [make() for _ in range(L)]
    vh = [make() for _ in range(L)]
    perm = torch.randperm(NB, generator=g).numpy()
    pairs = np.stack([perm[:8], perm[8:16]], axis=1).astype(np.int32)
    pairs = np.concatenate([pairs, [[NB, 3], [2, -1]]]).astype(np.int32)
    kd = [t.cuda() for t in kh]
    vd = [t.cuda() for t in vh]
    ks = [t.clone() for t in kd]
    vs = [t.clone() for t in vd]
    pd = torch.from_numpy(pairs).cuda()
    pkv.paged_copy_blocks_layers(kd, vd, pd)
    for l in range(L):
        pkv.paged_copy_blocks(ks[l], vs[l], pd)
    torch.cuda.synchronize()
    valid = pairs[(pairs >= 0).all(1) & (pairs < NB).all(1)]
    raw = lambda t: (t.view(torch.int16) if t.element_size() == 2 else t).cpu().numpy()
    for l in range(L):
        ko, vo = raw(kh[l]).copy(), raw(vh[l]).copy()
        cache_ops.copy_blocks(ko, vo, valid)
        assert np.array_equal(raw(kd[l]), ko)
        assert np.array_equal(raw(vd[l]), vo)
        assert np.array_equal(raw(kd[l]), raw(ks[l])) and np.array_equal(raw(vd[l]), raw(vs[l]))


def test_copy_blocks_layers_refusals():
    import paged_kv_cache_166_gb300 as pkv
    kc = [torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda") for _ in range(129)]
    pairs = torch.tensor([[0, 1]], dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError):
        pkv.paged_copy_blocks_layers(kc, kc, pairs)        # more than 128 layers
    with pytest.raises(ValueError):
        pkv.paged_copy_blocks_layers(kc[:2], kc[:1], pairs)  # K and V lists differ
    odd = torch.zeros(5, 2, 16, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        pkv.paged_copy_blocks_layers([kc[0], odd], [kc[1], kc[2]], pairs)
    pkv.paged_copy_blocks_layers(kc[:3], kc[3:6], pairs[:0])   # no pairs: nothing to do
    torch.cuda.synchronize()

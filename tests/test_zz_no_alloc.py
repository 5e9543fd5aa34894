"""The static-scratch decode entry point, for callers that cannot allocate.

Some callers cannot give the library a device workspace: serving engines that
hand all of HBM to the KV block pool at start-up and forbid later allocations,
plugins inside a framework that owns every device allocation, and decode loops
where cudaMalloc's implicit synchronisation is not acceptable.
pkv_decode_attention_static_scratch serves them from a fixed scratch array in
the library's device image.  This test calls it through the C ABI twice in a
row and checks each output against the fp64 oracle and against
pkv_decode_attention with a caller workspace, within the tolerance of the other
decode tests.  It also checks that requests the entry point must refuse (more
scratch than the array holds, or a head shape pkv_decode_attention refuses)
return their error and write nothing.  The file is named to run last, and passes
alone in a fresh process as well.
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


def call_static(b, tables, ctx, out, num_warps=0):
    from paged_kv_cache_166_gb300 import _native as N
    from paged_kv_cache_166_gb300.ops import dtype_code
    w = b.w
    S, Hq, D = b.q.shape
    NB, Hkv, B, _ = b.kc.shape
    return N.lib().pkv_decode_attention_static_scratch(
        b.q.data_ptr(), b.kc.data_ptr(), b.vc.data_ptr(), tables.data_ptr(), tables.shape[1],
        ctx.data_ptr(), S, Hq, Hkv, D, B, NB, float(w.scale), out.data_ptr(), num_warps,
        dtype_code(b.q), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,lens", [
    ("gqa70b", (1024, 5, 3000, 16, 17, 700, 1, 2100, 64, 250)),
    ("mha13b", (300, 1, 2048, 77, 16, 513, 129, 31)),
])
def test_static_scratch_matches_oracle_and_workspace_entry_point(name, lens):
    import paged_kv_cache_166_gb300 as pkv
    b = BT.decode_batch(W.WORKLOADS[name], np.asarray(lens))
    want = BT.oracle_rows(b, list(range(len(lens))))    # before the library writes the caches
    tables, ctx, slots = b.device_index("cuda")
    pkv.paged_kv_write(b.k_new, b.v_new, slots, b.kc, b.vc)
    ref = torch.empty_like(b.q)
    pkv.paged_decode_attention(b.q, b.kc, b.vc, tables, ctx, b.w.scale, ref)
    torch.cuda.synchronize()
    ref64 = BT.np64(ref)
    tol = BT.tolerance(b.w.dtype)
    for _ in range(2):
        out = torch.full_like(b.q, float("nan"))
        assert call_static(b, tables, ctx, out) == 0
        torch.cuda.synchronize()
        got = BT.np64(out)
        err = BT.row_errors(got, want)
        assert err.max() <= tol, err.max()
        err = BT.row_errors(got, ref64)
        assert err.max() <= tol, err.max()


def test_static_scratch_refuses_oversized_requests():
    from paged_kv_cache_166_gb300 import _native as N
    b = BT.decode_batch(W.WORKLOADS["gqa70b"], np.asarray((40, 3)))
    tables, ctx, _ = b.device_index("cuda")
    out = torch.zeros_like(b.q)
    rc = call_static(b, tables, ctx, out, num_warps=1 << 20)
    assert rc == N.PKV_ERR_UNSUPPORTED
    assert b"static scratch" in N.lib().pkv_last_error_string()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0


def test_static_scratch_refuses_what_the_workspace_entry_point_refuses():
    """12 query heads over 4 KV heads (groups of 3) is refused by the argument
    checks; nothing is written."""
    from paged_kv_cache_166_gb300 import _native as N
    from paged_kv_cache_166_gb300.ops import dtype_code
    b = BT.decode_batch(W.WORKLOADS["mha13b"], np.asarray((40, 3)))
    tables, ctx, _ = b.device_index("cuda")
    S, _, D = b.q.shape
    NB, Hkv, B, _ = b.kc.shape
    q = torch.zeros((S, 12, D), dtype=b.q.dtype, device="cuda")
    out = torch.full_like(q, 7.0)
    rc = N.lib().pkv_decode_attention_static_scratch(
        q.data_ptr(), b.kc.data_ptr(), b.vc.data_ptr(), tables.data_ptr(), tables.shape[1],
        ctx.data_ptr(), S, 12, 4, D, B, NB, float(b.w.scale), out.data_ptr(), 0,
        dtype_code(q), torch.cuda.current_stream().cuda_stream)
    assert rc == N.PKV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)

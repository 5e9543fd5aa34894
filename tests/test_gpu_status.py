"""Failure reporting on the device, without a fault.

Every kernel of the library waits on its mbarriers (TMA copies into shared memory,
tensor-core commits, hand-offs between warps) through one bounded wait that gives up
after a time limit, records PKV_DEV_WAIT_TIMEOUT and lets the kernel return.  Here
that wait is made to run out on purpose: pkv_wait_timeout_selftest waits on an
mbarrier that nothing completes.  The test checks that the wait ends after its limit,
that the status bit reaches the host, that a completed phase is then seen at once,
and that the context stays usable: a decode launch right after it still matches the
fp64 oracle.
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


@pytest.mark.parametrize("limit_us", [2000, 20000])
def test_bounded_wait_runs_out_and_reports(limit_us):
    import paged_kv_cache_166_gb300 as pkv
    from paged_kv_cache_166_gb300 import _native as N
    status, waited_ns, then_ok = pkv.wait_timeout_selftest(limit_us)
    assert status == N.PKV_DEV_WAIT_TIMEOUT
    assert waited_ns >= limit_us * 1000
    assert waited_ns < limit_us * 1000 + 500_000_000  # gave up, did not hang on
    assert then_ok


def test_context_usable_after_a_wait_ran_out():
    import paged_kv_cache_166_gb300 as pkv
    from paged_kv_cache_166_gb300 import _native as N
    status, _, _ = pkv.wait_timeout_selftest(5000)
    assert status == N.PKV_DEV_WAIT_TIMEOUT
    lens = np.asarray((300, 1, 2048, 77, 16, 513))
    b = BT.decode_batch(W.WORKLOADS["gqa70b"], lens)
    want = BT.oracle_rows(b, list(range(len(lens))))
    tables, ctx, slots = b.device_index("cuda")
    pkv.paged_kv_write(b.k_new, b.v_new, slots, b.kc, b.vc)
    out = torch.full_like(b.q, float("nan"))
    ws = torch.zeros(pkv.workspace_bytes(b.q.shape[1], b.kc.shape[1], b.q.shape[2], b.q.dtype),
                     dtype=torch.uint8, device="cuda")
    pkv.paged_decode_attention(b.q, b.kc, b.vc, tables, ctx, b.w.scale, out, ws)
    torch.cuda.synchronize()
    assert pkv.decode_status(ws) == 0
    err = BT.row_errors(BT.np64(out), want)
    assert err.max() <= BT.tolerance(b.w.dtype), err.max()

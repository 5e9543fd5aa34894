"""The product path has no CPU fallback and fails loudly (no GPU needed).

* Without libpkv.so every entry of the binding raises, naming the missing library;
  nothing computes on the CPU instead.
* The torch-facing ops refuse host tensors before any call reaches the library.
"""
import subprocess
import sys

import pytest
import torch

from conftest import ROOT


def test_missing_library_raises_instead_of_falling_back(tmp_path):
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from paged_kv_cache_166_gb300 import _native as N\n"
        "N.LIB_PATH = %r\n"
        "import paged_kv_cache_166_gb300 as pkv\n"
        "for call in (lambda: N.lib(), lambda: pkv.BlockAllocator(8, 16)):\n"
        "    try:\n"
        "        call()\n"
        "    except RuntimeError as e:\n"
        "        assert 'is not built' in str(e), e\n"
        "    else:\n"
        "        raise SystemExit('no error without the library')\n"
        "print('raised')\n" % (ROOT, str(tmp_path / "libpkv.so")))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("raised")


def _host_case():
    S, Hq, Hkv, D, NB, B = 2, 4, 4, 64, 8, 16
    q = torch.zeros(S, Hq, D, dtype=torch.float16)
    kc = torch.zeros(NB, Hkv, B, D, dtype=torch.float16)
    tables = torch.zeros(S, 2, dtype=torch.int32)
    ctx = torch.ones(S, dtype=torch.int32)
    return q, kc, tables, ctx


def test_ops_refuse_host_tensors():
    import paged_kv_cache_166_gb300 as pkv
    q, kc, tables, ctx = _host_case()
    out = torch.full_like(q, 7.0)
    kn = torch.zeros(q.shape[0], kc.shape[1], q.shape[2], dtype=q.dtype)
    calls = [
        lambda: pkv.paged_decode_attention(q, kc, kc.clone(), tables, ctx, 0.125, out),
        lambda: pkv.paged_decode_step(q, kn, kn.clone(), kc, kc.clone(), tables, ctx, 0.125, out),
        lambda: pkv.paged_kv_write(kn, kn.clone(), torch.zeros(2, dtype=torch.int32), kc,
                                   kc.clone()),
        lambda: pkv.paged_prefill_attention(q, kc, kc.clone(), tables, ctx,
                                            torch.tensor([0, 1, 2], dtype=torch.int32), 0.125,
                                            out),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensors"):
            call()
    assert torch.all(out == 7.0)  # nothing was computed on the host instead

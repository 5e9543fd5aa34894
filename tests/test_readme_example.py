"""The README's Python usage example stays in step with the binding (no GPU needed).

The example is taken from README.md and run on the host with its device set to the
CPU and every torch-facing op replaced by a stand-in that only binds the call's
arguments to the real op's signature: the block-manager calls run for real, and a
call with a wrong name or argument list fails here.
"""
import inspect
import os
import re

from conftest import ROOT


def test_readme_example_calls_match_the_binding(monkeypatch):
    from paged_kv_cache_166_gb300 import ops
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) == 1
    code = blocks[0].replace('dev = "cuda"', 'dev = "cpu"')
    assert 'dev = "cpu"' in code
    called = []
    for name in [n for n in dir(ops) if n.startswith("paged_")]:
        real = getattr(ops, name)

        def stand_in(*args, _real=real, _name=name, **kw):
            inspect.signature(_real).bind(*args, **kw)
            called.append(_name)

        monkeypatch.setattr(ops, name, stand_in)
    exec(compile(code, "README.md example", "exec"), {"__name__": "readme_example"})
    assert called == ["paged_kv_write", "paged_prefill_attention", "paged_copy_blocks",
                      "paged_decode_step"]

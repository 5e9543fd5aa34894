"""Host logic of bench.py that needs no GPU: the comment-free code hash that ties
an ncu summary to the kernel source it was captured from, and the summaries'
figures as bench.py reads them."""
import glob
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_sha_ignores_comments_and_whitespace_only():
    a = "int f(int x) {  // doubles\n  return 2 * x; /* the\n result */\n}\n"
    b = "int f(int x) {\n\n  return 2 * x;   // twice x\n}"
    c = "int f(int x) {\n  return 3 * x;\n}"
    assert bench.code_sha(a) == bench.code_sha(b)
    assert bench.code_sha(a) != bench.code_sha(c)
    assert len(bench.code_sha(a)) == 16


def test_every_profile_summary_parses_and_names_its_capture():
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", "*_attention_*.md")) +
                   glob.glob(os.path.join(ROOT, "profiles", "kv_write_*.md")))
    assert paths
    for p in paths:
        fields = dict(l.strip("- ").split(": ", 1) for l in open(p).read().splitlines()
                      if l.startswith("- ") and ": " in l)
        assert len(fields["source_sha"]) == 16 and len(fields["code_sha"]) == 16, p
        assert int(fields["traffic_bytes_per_launch"]) > 0, p
        tag = os.path.basename(p)[:-3]
        src = ("prefill_tcgen05.cu" if tag.startswith("prefill") else
               "kv_ops.cu" if tag.startswith("kv_write") else "decode_attention.cu")
        got = bench.profile_traffic(tag, src, fields.get("workload_key"))
        # the figure is reported exactly when the kernel's code is the captured one
        text = open(os.path.join(ROOT, "paged_kv_cache_166_gb300", "csrc", src)).read()
        same = bench.code_sha(text) == fields["code_sha"]
        assert (got == int(fields["traffic_bytes_per_launch"])) if same else got is None, p


def _ref_args(**kw):
    import types
    a = dict(workload="tiny", steps=2, warmup=3, ref_budget=0.5)
    a.update(kw)
    return types.SimpleNamespace(**a)


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.reference(_ref_args())
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    """The oracle arm's JSON line on the small workload: its own cpu_baseline and an
    e2e with no host-device bytes, every pass over one bounded sample."""
    import json
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.reference(_ref_args())
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert "4 of 4 sequences" in line["cpu_baseline"]["sample"]

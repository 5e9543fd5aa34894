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
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", "*_attention_*.md")))
    assert paths
    for p in paths:
        fields = dict(l.strip("- ").split(": ", 1) for l in open(p).read().splitlines()
                      if l.startswith("- ") and ": " in l)
        assert len(fields["source_sha"]) == 16 and len(fields["code_sha"]) == 16, p
        assert int(fields["traffic_bytes_per_launch"]) > 0, p
        tag = os.path.basename(p)[:-3]
        src = "prefill_tcgen05.cu" if tag.startswith("prefill") else "decode_attention.cu"
        got = bench.profile_traffic(tag, src, fields.get("workload_key"))
        # the figure is reported exactly when the kernel's code is the captured one
        text = open(os.path.join(ROOT, "paged_kv_cache_166_gb300", "csrc", src)).read()
        same = bench.code_sha(text) == fields["code_sha"]
        assert (got == int(fields["traffic_bytes_per_launch"])) if same else got is None, p

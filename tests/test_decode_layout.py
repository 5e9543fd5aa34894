"""The decode kernel's shared-memory layout (csrc/decode_layout.h), checked on the
CPU: for every batch size the kernel takes (1..2048 sequences), every warp count per
CTA, pipeline depth, query-slot stride and stage size the launcher can pick, every
region starts on the boundary its accesses need (TMA tiles 1024 B, bulk-copied
query slots 16 B, mbarriers 8 B, words 4 B) and regions do not overlap.  A
misaligned region faults the GPU; this pins the layout without one."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_cache_166_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "decode_layout.h"
using namespace pkv;
int main() {
  long checked = 0;
  const int stage_bytes[] = {4096, 8192, 16384};
  const int q_strides[] = {0, 128, 256, 512, 1024, 2048, 4096};
  const int warps[] = {4, 8, 16};
  for (int S = 1; S <= 2048; ++S)
    for (int sb : stage_bytes)
      for (int qs : q_strides)
        for (int nw : warps)
          for (int st = 0; st <= 12; ++st)
            {
              const SmemLayout L = smem_layout(sb, st, qs, S, nw);
              const bool order = L.tiles <= L.q && L.q <= L.bars && L.bars <= L.ids &&
                                 L.ids + nw * 512u <= L.ctx && L.ctx + 4u * S <= L.pre &&
                                 L.pre + 4u * (S + 1) <= L.prew &&
                                 L.prew + 4u * (S + 1) <= L.scratch &&
                                 L.scratch + 256u + 1024u <= L.total;
              if (!smem_layout_aligned(L, sb, qs) || !order) {
                std::printf("bad layout S=%d stage=%d q=%d nw=%d stages=%d\n", S, sb, qs, nw, st);
                return 1;
              }
              ++checked;
            }
  std::printf("%ld layouts aligned\n", checked);
  return 0;
}
"""


def test_every_layout_is_aligned(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "layout.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "layout"
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "layouts aligned" in out.stdout


def test_a_misplaced_region_is_caught(tmp_path):
    """The pin fails on the kind of layout that faulted once: a byte-sized
    per-sequence region (S bytes) placed before word-sized ones, which leaves them
    off their boundary whenever S is not a multiple of the word size."""
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    header = open(os.path.join(CSRC, "decode_layout.h")).read()
    old = "  L.pre = off;"
    assert old in header
    (tmp_path / "decode_layout.h").write_text(header.replace(old, "  off += S;\n  L.pre = off;"))
    src = tmp_path / "layout.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "layout"
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", str(tmp_path), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 1 and "bad layout S=1 " in out.stdout

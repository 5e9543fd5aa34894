"""Host-side tests of the C ABI (no GPU needed).

* libpkv.so loads without a GPU and exports every function include/pkv.h declares,
  each with a ctypes signature in the binding whose arguments match the prototype
  kind for kind; the header compiles as strict C99 and a C program links and runs
  against the library.
* The library's block manager matches the oracle model bit for bit — tables,
  lengths, slots, copy-on-write pairs, refcounts and free counts after every
  operation — on the pages' worked examples and on seeded random operation
  sequences; failing calls leave both unchanged.
"""
import os
import re

import numpy as np
import pytest

from conftest import ROOT
from oracle.block_manager import BlockManager, InvalidOperation, OutOfBlocks as OracleOOB

pkv = pytest.importorskip("paged_kv_cache_166_gb300")
from paged_kv_cache_166_gb300 import _native as N  # noqa: E402
from paged_kv_cache_166_gb300 import BlockAllocator  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def header_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = header_functions()
    assert len(names) >= 20
    lib = N.lib()
    for name in names:
        assert hasattr(lib, name), name
        assert name in N.SIGNATURES, f"no binding signature for {name}"
    assert set(N.SIGNATURES) == set(names)
    assert lib.pkv_version() >= 100


def _c_kind(param: str) -> str:
    param = " ".join(param.split())
    if "*" in param:
        return "ptr"
    for ctype, kind in (("int32_t", "i32"), ("int64_t", "i64"), ("size_t", "size"),
                        ("float", "f32"), ("int", "i32"), ("char", "char")):
        if re.search(r"\b" + ctype + r"\b", param):
            return kind
    return "unknown: " + param


def _ctypes_kind(t) -> str:
    import ctypes
    if t in (ctypes.c_void_p, ctypes.c_char_p) or (isinstance(t, type) and
                                                   issubclass(t, ctypes._Pointer)):
        return "ptr"
    return {ctypes.c_int32: "i32", ctypes.c_int64: "i64", ctypes.c_size_t: "size",
            ctypes.c_float: "f32"}.get(t, f"unknown: {t}")


def _signature_mismatches(signatures) -> list:
    """(name, header kinds, binding kinds) for every prototype of include/pkv.h whose
    ctypes declaration differs in argument count, an argument's kind (pointer, int32,
    int64, size_t, float) or the return kind."""
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"#[^\n]*", "", text)
    protos = re.findall(r"([A-Za-z_][A-Za-z_0-9 *]*?)\b(pkv_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;",
                        text, flags=re.S)
    assert sorted(name for _, name, _ in protos) == header_functions()
    bad = []
    for ret, name, params in protos:
        args = [p.strip() for p in params.split(",") if p.strip() and p.strip() != "void"]
        restype, argtypes = signatures[name]
        want = [_c_kind(ret)] + [_c_kind(p) for p in args]
        got = [_ctypes_kind(restype)] + [_ctypes_kind(t) for t in argtypes]
        if want != got:
            bad.append((name, want, got))
    return bad


def test_binding_signatures_match_the_header():
    """A misdeclared argument would otherwise pass a wrong value silently."""
    assert _signature_mismatches(N.SIGNATURES) == []
    # planted: one argument dropped, one int32 declared as int64
    import ctypes
    planted = dict(N.SIGNATURES)
    ret, args = planted["pkv_kv_write"]
    planted["pkv_kv_write"] = (ret, args[:-1])
    ret, args = planted["pkv_copy_blocks"]
    planted["pkv_copy_blocks"] = (ret, [args[0], args[1], args[2], ctypes.c_int64] + args[4:])
    assert [b[0] for b in _signature_mismatches(planted)] == ["pkv_kv_write", "pkv_copy_blocks"]


def test_error_codes_and_messages_without_gpu():
    lib = N.lib()
    import ctypes
    n = ctypes.c_size_t()
    assert lib.pkv_decode_workspace_size(6, 4, 128, N.PKV_BF16, 8, ctypes.byref(n)) == N.PKV_ERR_INVALID_ARG
    assert b"head counts" in lib.pkv_last_error_string()
    assert lib.pkv_decode_workspace_size(8, 1, 128, 9, 8, ctypes.byref(n)) == N.PKV_ERR_DTYPE
    assert lib.pkv_decode_workspace_size(8, 1, 96, N.PKV_BF16, 8, ctypes.byref(n)) == N.PKV_ERR_UNSUPPORTED
    assert lib.pkv_decode_workspace_size(8, 1, 128, N.PKV_BF16, 8, ctypes.byref(n)) == N.PKV_OK
    # status word, 8 tickets, m/l and accumulator partials of 2 pieces per warp
    assert n.value == 256 + 256 + 2 * 8 * 8 * 2 * 4 + 2 * 8 * 8 * 128 * 4
    assert lib.pkv_kv_write(None, None, None, 0, None, None, 4, 2, 16, 100, N.PKV_F16, None) == N.PKV_ERR_INVALID_ARG
    # the bounded-wait self-test checks its arguments before it launches anything
    assert lib.pkv_wait_timeout_selftest(None, None, 1000, None) == N.PKV_ERR_INVALID_ARG
    for limit in (0, -5, 1000001):
        assert lib.pkv_wait_timeout_selftest(64, 128, limit, None) == N.PKV_ERR_INVALID_ARG
        assert b"limit_us" in lib.pkv_last_error_string()
    assert lib.pkv_wait_timeout_selftest(66, 128, 1000, None) == N.PKV_ERR_INVALID_ARG


class Pair:
    """Drives the library's block manager and the oracle model with the same operations."""

    def __init__(self, nb, bs, order=None):
        self.c = BlockAllocator(nb, bs, order)
        self.o = BlockManager(nb, bs, order)
        self.nb = nb

    def compare(self):
        for b in range(self.nb):
            assert self.c.refcount(b) == self.o.refcount[b]
        assert self.c.num_free() == self.o.num_free()
        for sid in self.o.tables:
            assert self.c.table(sid) == self.o.tables[sid]
            assert self.c.length(sid) == self.o.lengths[sid]

    def create(self):
        a, b = self.c.create(), self.o.create()
        assert a == b
        return a

    def fork(self, p):
        a, b = self.c.fork(p), self.o.fork(p)
        assert a == b
        return a

    def free(self, s):
        self.c.free(s)
        self.o.free(s)

    def swap_out(self, s):
        a, b = self.c.swap_out(s), self.o.swap_out(s)
        assert a == b
        return a

    def swap_in(self, s):
        try:
            b = self.o.swap_in(s)
        except OracleOOB:
            with pytest.raises(N.OutOfBlocks):
                self.c.swap_in(s)
            return None
        a = self.c.swap_in(s)
        assert a == b
        return a

    def append(self, s, n):
        need = self.o.blocks_needed(s, n)
        assert self.c.blocks_needed(s, n) == need
        try:
            so, co = self.o.append(s, n)
        except OracleOOB:
            with pytest.raises(N.OutOfBlocks):
                self.c.append(s, n)
            return None
        sc, cc = self.c.append(s, n)
        assert list(sc) == so
        assert cc == co
        return so, co


def test_worked_example_matches_oracle(golden):
    from test_oracle_block_manager import run_script
    run_script(golden("worked_example_b4.txt"), BlockAllocatorView)


class BlockAllocatorView:
    """Adapter exposing the oracle's attribute view on top of the library handle."""

    def __init__(self, nb, bs):
        self.a = BlockAllocator(nb, bs)
        self.nb = nb
        self.live = set()

    def create(self):
        s = self.a.create(); self.live.add(s); return s

    def fork(self, p):
        s = self.a.fork(p); self.live.add(s); return s

    def free(self, s):
        self.a.free(s); self.live.discard(s)

    def append(self, s, n):
        slots, cows = self.a.append(s, n)
        return list(slots), cows

    def num_free(self):
        return self.a.num_free()

    @property
    def tables(self):
        return {s: self.a.table(s) for s in self.live}

    @property
    def refcount(self):
        return [self.a.refcount(b) for b in range(self.nb)]


def test_eight_requests_and_parallel_sampling_match_oracle():
    p = Pair(3072, 16)
    for length in (180, 220, 260, 310, 400, 520, 1400, 1900):
        s = p.create()
        p.append(s, length)
    p.compare()
    assert p.c.num_free() == 2744
    q = Pair(1000, 16)
    parent = q.create()
    q.append(parent, 1000)
    kids = [q.fork(parent) for _ in range(3)]
    for s in [parent] + kids:
        q.append(s, 200)
    q.compare()
    assert 1000 - q.c.num_free() == 114


@pytest.mark.parametrize("seed", range(8))
def test_random_operations_bit_exact(seed):
    r = np.random.default_rng(seed)
    B = int(r.choice([1, 2, 4, 16]))
    NB = int(r.integers(8, 96))
    p = Pair(NB, B, r.permutation(NB).astype(np.int32))
    live, swapped = [], []
    for _ in range(600):
        op = r.integers(0, 12)
        if op < 2 or not live:
            live.append(p.create())
        elif op < 7:
            p.append(live[r.integers(len(live))], int(r.integers(0, 3 * B + 2)))
        elif op < 8:
            live.append(p.fork(live[r.integers(len(live))]))
        elif op < 9:
            p.free(live.pop(r.integers(len(live))))
        elif op < 10:
            swapped.append(live.pop(r.integers(len(live))))
            p.swap_out(swapped[-1])
        elif swapped:
            s = swapped[r.integers(len(swapped))]
            if p.swap_in(s) is not None:
                swapped.remove(s)
                live.append(s)
        p.compare()
    for s in swapped:  # swapped-out sequences refuse resident operations
        with pytest.raises(N.PkvError):
            p.c.append(s, 1)
        with pytest.raises(N.PkvError):
            p.c.fork(s)


def test_export_tables_matches_oracle():
    p = Pair(64, 4, np.random.default_rng(3).permutation(64).astype(np.int32))
    seqs = [p.create() for _ in range(5)]
    for i, s in enumerate(seqs):
        p.append(s, 3 * i + 1)
    kid = p.fork(seqs[3])
    p.append(kid, 2)
    order = [kid, seqs[0], seqs[4]]
    tc, cc = p.c.export_tables(order, 6)
    to, co = p.o.export_tables(order, 6)
    assert np.array_equal(tc, to) and np.array_equal(cc, co)
    with pytest.raises(N.PkvError):
        p.c.export_tables(order, 2)


def test_library_rejects_bad_operations_without_state_change():
    a = BlockAllocator(4, 4)
    s = a.create()
    a.append(s, 16)
    with pytest.raises(N.OutOfBlocks):
        a.append(s, 1)
    assert a.length(s) == 16 and a.num_free() == 0
    with pytest.raises(N.PkvError):
        a.decref(99)
    with pytest.raises(N.PkvError):
        a.free(7)
    with pytest.raises(N.PkvError):
        BlockAllocator(4, 4, pop_order=[0, 1, 1, 2])
    a.free(s)
    assert a.num_free() == 4
    with pytest.raises(N.PkvError):
        a.free(s)
    with pytest.raises(N.PkvError):
        a.incref(0)


@pytest.mark.parametrize("seed", range(6))
def test_append_one_each_equals_appends_in_list_order(seed):
    """pkv_seq_append_one_each against the oracle's block manager appending one
    token to each listed sequence in turn: the same slots, the same copy-on-write
    pairs in list order, the same state afterwards; when the pool cannot serve all
    of them, PKV_ERR_OUT_OF_BLOCKS and no change at all.  Forked siblings put
    shared partial blocks in the lists (the last holder writes in place)."""
    import copy
    r = np.random.default_rng(100 + seed)
    B = int(r.choice([2, 4, 16]))
    NB = int(r.integers(16, 80))
    p = Pair(NB, B, r.permutation(NB).astype(np.int32))
    live = []
    for _ in range(300):
        op = r.integers(0, 10)
        if op < 2 or not live:
            live.append(p.create())
        elif op < 4:
            p.append(live[r.integers(len(live))], int(r.integers(0, 2 * B + 2)))
        elif op < 5:
            live.append(p.fork(live[r.integers(len(live))]))
        elif op < 6 and len(live) > 1:
            p.free(live.pop(r.integers(len(live))))
        else:
            k = int(r.integers(0, len(live) + 1))
            seqs = [live[i] for i in r.permutation(len(live))[:k]]
            trial = copy.deepcopy(p.o)
            try:
                expect = [trial.append(s, 1) for s in seqs]
            except OracleOOB:
                before = p.c.num_free()
                with pytest.raises(N.OutOfBlocks):
                    p.c.append_one_each(seqs)
                assert p.c.num_free() == before
            else:
                slots, cows = p.c.append_one_each(seqs)
                assert list(slots) == [e[0][0] for e in expect]
                assert cows == [c for e in expect for c in e[1]]
                p.o = trial
        p.compare()
    if live:
        with pytest.raises(N.PkvError):  # an id listed twice
            p.c.append_one_each([live[0], live[0]])
    if len(live) >= 2:
        before = p.c.num_free()
        with pytest.raises(N.PkvError):  # listed twice, not side by side: nothing changes
            p.c.append_one_each([live[0], live[1], live[0]])
        assert p.c.num_free() == before
        p.compare()
        # the refused call leaves no trace: the same ids once each behave as appends
        trial = copy.deepcopy(p.o)
        try:
            expect = [trial.append(s, 1) for s in (live[1], live[0])]
        except OracleOOB:
            with pytest.raises(N.OutOfBlocks):
                p.c.append_one_each([live[1], live[0]])
        else:
            slots, cows = p.c.append_one_each([live[1], live[0]])
            assert list(slots) == [e[0][0] for e in expect]
            assert cows == [c for e in expect for c in e[1]]
            p.o = trial
        p.compare()
    with pytest.raises(N.PkvError):  # an unknown id
        p.c.append_one_each([10 ** 6])
    slots, cows = p.c.append_one_each([])
    assert len(slots) == 0 and cows == []


def test_decode_step_tables_equal_the_oracle_decode_loop():
    """DecodeStepTables (one new position per sequence, then the tables exported into
    caller-owned arrays, all arguments bound once) against the oracle's block manager
    appending one token to each sequence and reading its tables: the same slots,
    copy-on-write pairs, tables and lengths at every step of a decode loop with forked
    siblings sharing partial blocks."""
    from paged_kv_cache_166_gb300 import DecodeStepTables
    r = np.random.default_rng(11)
    B, NB = 4, 200
    p = Pair(NB, B, r.permutation(NB).astype(np.int32))
    seqs = []
    for t in (1, 6, 9, 4):
        s = p.create()
        p.append(s, t)
        seqs.append(s)
    seqs.append(p.fork(seqs[1]))      # shares a partial block with its parent
    seqs.append(p.fork(seqs[2]))
    maxb = 12
    tab = np.full((len(seqs), maxb), -7, dtype=np.int32)
    ctx = np.full(len(seqs), -7, dtype=np.int32)
    step = DecodeStepTables(p.c, seqs, maxb, tab, ctx)
    for _ in range(20):
        expect = [p.o.append(s, 1) for s in seqs]
        slots, cows = step()
        assert list(slots) == [e[0][0] for e in expect]
        assert cows == [c for e in expect for c in e[1]]
        for i, s in enumerate(seqs):
            t = p.o.tables[s]
            assert list(tab[i, :len(t)]) == list(t) and not tab[i, len(t):].any()
            assert ctx[i] == p.o.lengths[s]
        p.compare()
    with pytest.raises(ValueError):
        DecodeStepTables(p.c, seqs, maxb, tab[:, :3].copy(), ctx)


def test_header_is_plain_c_and_links_against_the_library(tmp_path):
    """include/pkv.h compiles as strict C99 and every function it declares resolves
    against libpkv.so at link time; the program then drives the block manager through
    the C ABI alone (no Python in between)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = header_functions()
    table = ",\n".join(f"  (void (*)(void))&{n}" for n in names)
    src = tmp_path / "abi.c"
    src.write_text(f"""#include <stdio.h>
#include "pkv.h"
static void (*const fns[])(void) = {{
{table}
}};
int main(void) {{
  pkv_allocator_t* a = 0;
  int32_t s = -1, slots[20], cow[2], ncow = -1, nfree = -1;
  if (pkv_allocator_create(4, 16, 0, &a) != PKV_OK) return 1;
  if (pkv_seq_create(a, &s) != PKV_OK) return 2;
  if (pkv_seq_append(a, s, 20, slots, cow, &ncow) != PKV_OK || ncow != 0) return 3;
  if (slots[0] != 0 || slots[15] != 15 || slots[16] != 16 || slots[19] != 19) return 4;
  if (pkv_num_free_blocks(a, &nfree) != PKV_OK || nfree != 2) return 5;
  if (pkv_seq_append(a, 99, 1, slots, cow, &ncow) == PKV_OK) return 6;
  pkv_allocator_destroy(a);
  printf("%d\\n", (int)(sizeof(fns) / sizeof(fns[0])));
  return 0;
}}
""")
    lib = os.path.join(ROOT, "paged_kv_cache_166_gb300", "libpkv.so")
    exe = tmp_path / "abi"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), lib,
                    "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out
    assert int(out.stdout) == len(names)

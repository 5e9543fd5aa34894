"""Benchmark of one decode step of the paged KV-cache hot path on GB300.

A step is one pass of the whole hot path over one batch, through one call of
the decode step: the cache write of every sequence's new token (into the slot
the library's block manager gave its position) and paged decode attention over
all cached tokens, new token included; split contexts are merged inside the
attention launch.  The two launches are chained with programmatic dependent
launch.

Default workload: the 13B-shaped MHA decode batch (64 sequences, 40 query = 40
KV heads, head_dim 128, fp16, block size 16, lognormal lengths with median 300
and sigma 1.0 clipped to [1, 2048], pool = blocks + 10% shuffled).

value     = algorithmic KV-read bytes of decode attention / device step time
            (CUDA events on the launching stream; L2 flushed between steps).
e2e       = the same bytes / end-to-end layer-step time of a decode loop through
            the public API over a two-layer model: every token step runs the host
            block manager, one H2D copy of both layers' packed q and new K/V with the
            tables and lengths from page-locked memory, the decode step on each
            layer's cache and the D2H copies of the outputs; the host prepares the
            next token step while the device runs the current one (the
            one-step-at-a-time figures are reported beside it).
roofline  = the decode-attention kernel, the dominant launch of a step (timed
            in its own loop, L2 flushed): its algorithmic bytes / its event time,
            against the measured HBM copy bandwidth.
cpu_baseline / --impl reference = the fp64 oracle on the host cores.

Under torchrun with N ranks each rank runs an independent replica of the
workload on its own GPU (the path shards by sequence with no exchange step);
value = bytes of all ranks / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attn KV-read GB/s (% of GB300 HBM peak); seq-tokens/s per layer"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20  # > 129 MB L2


class L2Flush:
    """Between timed steps: writes a buffer larger than L2, then reads another as
    large, so that the next launch finds neither its inputs in L2 nor dirty lines of
    the flush buffer that it would have to write back to DRAM on its own clock."""

    LABEL = f"flushed between steps ({FLUSH_BYTES >> 20} MiB write, then {FLUSH_BYTES >> 20} MiB read, untimed)"

    def __init__(self, device):
        import torch
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def attention_bytes(lens, Hq, Hkv, D, elt, B=16, q_elt=None) -> int:
    """Algorithmic bytes decode attention must move: K and V rows of the cached
    tokens (no padded block tails, `elt` bytes per element), the int32 table
    entries, the context length, one query and one output row per query head
    (`q_elt` bytes per element, default `elt`)."""
    lens = np.asarray(lens, dtype=np.int64)
    nb = (lens + B - 1) // B
    q_elt = elt if q_elt is None else q_elt
    return int((2 * lens * Hkv * D * elt + 4 * nb + 4 + 2 * Hq * D * q_elt).sum())


def kv_write_bytes(num_tokens, Hkv, D, elt) -> int:
    return int(num_tokens * (2 * 2 * Hkv * D * elt + 4))


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def max_over_ranks(values, device=None):
    """Element-wise maximum of `values` over all ranks of the default process
    group (the values themselves without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_gbs(bytes_per_rank: int, world: int, ms: float) -> float:
    """Throughput of the whole job: every rank moves bytes_per_rank in its step,
    the job's step lasts as long as its slowest rank (ms)."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


def code_sha(text: str) -> str:
    """First 16 hex digits of sha256 of a C++/CUDA source with its comments removed
    and its whitespace collapsed: unchanged by edits to comments alone."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


def profile_traffic(kernel_tag: str, source: str = "decode_attention.cu", workload_key=None):
    """Per-launch DRAM bytes from the committed ncu summary of this kernel, if the
    kernel's code is unchanged since it was captured (the summary's code_sha, else
    its whole-file source_sha) and, when given, the summary was taken on the same
    workload."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    src = os.path.join(ROOT, "paged_kv_cache_166_gb300", "csrc", source)
    try:
        text = open(path).read()
        raw = open(src, "rb").read()
        fields = dict(l.strip("- ").split(": ", 1) for l in text.splitlines()
                      if l.startswith("- ") and ": " in l)
        if "code_sha" in fields:
            if fields["code_sha"] != code_sha(raw.decode()):
                return None
        elif fields.get("source_sha") != hashlib.sha256(raw).hexdigest()[:16]:
            return None
        if workload_key is not None and fields.get("workload_key") != workload_key:
            return None
        return int(fields["traffic_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, name):
        setattr(self, name, time.perf_counter())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        """Median SM clock and throttle reasons of the samples taken in [t0, t1]."""
        if not self.lines:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, l in self.lines:
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------------------
# workload construction through the library (block manager -> tables, slots)
# --------------------------------------------------------------------------------------
def workload_config(w, lens, NB: int, q8=None) -> dict:
    """The workload keys of a decode line's config (the same for both arms)."""
    kv_name = {"fp8": "fp8 (E4M3)", "int8": "int8"}.get(q8)
    S, Hq, Hkv, D, B = len(lens), w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    return {
        "workload": f"{w.name}: {S} seqs, {Hq} q / {Hkv} kv heads, head_dim {D}, {w.dtype}, "
                    f"block {B}, lengths sum {int(lens.sum())} max {int(lens.max())}, pool {NB} blocks"
                    + (f", {kv_name} KV cache with per-KV-head scales" if q8 else ""),
        "num_seqs": S, "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": D,
        "block_size": B, "sum_context": int(lens.sum()), "num_blocks": NB,
        "kv_cache": {"fp8": "fp8 e4m3", "int8": "int8"}.get(q8, w.dtype),
    }


def pool_blocks(w, lens) -> int:
    B = w.block_size
    blocks = int(((lens + B - 1) // B).sum())
    return w.fixed_pool_blocks or int(math.ceil(blocks * (1 + w.pool_spare))) + 1


def build_batch(name: str, device, rank: int = 0, kv: str = "native", block_size: int = 0,
                grow_tokens: int = 0):
    """The decode batch of a workload on `device`, its tables built by the library's
    block manager (history of ctx - 1 tokens per sequence, then the new token).

    grow_tokens > 0 reserves blocks past the workload's pool for a decode loop that
    appends that many more tokens to every sequence; they are handed out only after
    the pool's own ids, so the workload's tables are the same either way.  Returns
    (w, lens, NB, kc, vc, host, dev, alloc, sids) with NB the workload's pool."""
    import torch
    from paged_kv_cache_166_gb300 import BlockAllocator
    from paged_kv_cache_166_gb300 import workloads as W

    w = W.WORKLOADS[name]
    if block_size and block_size != w.block_size:
        import dataclasses
        w = dataclasses.replace(w, block_size=block_size)
    seed = w.seed + 1000 * rank
    lens = W.context_lengths(w)
    if rank:
        import dataclasses
        lens = W.context_lengths(dataclasses.replace(w, seed=seed)) if w.length_kind != "fixed" else lens
    B = w.block_size
    NB = pool_blocks(w, lens)
    order = W.pool_order(NB, seed)
    extra = len(lens) * (grow_tokens // B + 2) if grow_tokens > 0 else 0
    if extra:
        order = np.concatenate([order, np.arange(NB, NB + extra, dtype=np.int32)])
    alloc = BlockAllocator(NB + extra, B, order)
    sids = [alloc.create() for _ in range(len(lens))]
    for s, t in zip(sids, lens):
        alloc.append(s, int(t) - 1)
    new_slots = np.array([alloc.append(s, 1)[0][0] for s in sids], dtype=np.int32)
    maxb = int(((lens + B - 1) // B).max())
    tables, ctx = alloc.export_tables(sids, maxb)
    dt = W.torch_dtype(w.dtype)
    S, Hq, Hkv, D = len(lens), w.num_q_heads, w.num_kv_heads, w.head_dim
    if kv == "fp8":
        # E4M3 codes of N(0,1) draws with per-KV-head scales; V tiles transposed
        kc = torch.empty((NB + extra, Hkv, B, D), dtype=torch.uint8, device=device)
        vc = torch.empty((NB + extra, Hkv, D, B), dtype=torch.uint8, device=device)
        k_scale, v_scale = W.fp8_scales(Hkv, seed), W.fp8_scales(Hkv, seed + 1)
        W.fill_fp8_codes_(kc, k_scale, seed, W.STREAM_K_POOL)
        W.fill_fp8_codes_(vc, v_scale, seed, W.STREAM_V_POOL)
    elif kv == "int8":
        # int8 codes of N(0,1) draws with per-KV-head scales; V tiles transposed
        kc = torch.empty((NB + extra, Hkv, B, D), dtype=torch.int8, device=device)
        vc = torch.empty((NB + extra, Hkv, D, B), dtype=torch.int8, device=device)
        k_scale, v_scale = W.int8_scales(Hkv, seed), W.int8_scales(Hkv, seed + 1)
        W.fill_int8_codes_(kc, k_scale, seed, W.STREAM_K_POOL)
        W.fill_int8_codes_(vc, v_scale, seed, W.STREAM_V_POOL)
    else:
        kc = torch.empty((NB + extra, Hkv, B, D), dtype=dt, device=device)
        vc = torch.empty_like(kc)
        W.fill_normal_(kc, seed, W.STREAM_K_POOL)
        W.fill_normal_(vc, seed, W.STREAM_V_POOL)
    host = {
        "q": W.normal_tensor((S, Hq, D), w.dtype, seed, W.STREAM_Q, "cpu"),
        "k_new": W.normal_tensor((S, Hkv, D), w.dtype, seed, W.STREAM_K_NEW, "cpu"),
        "v_new": W.normal_tensor((S, Hkv, D), w.dtype, seed, W.STREAM_V_NEW, "cpu"),
        "slots": torch.from_numpy(new_slots),
        "tables": torch.from_numpy(tables),
        "ctx": torch.from_numpy(ctx),
    }
    host = {k: v.pin_memory() for k, v in host.items()}
    dev = {k: v.to(device) for k, v in host.items()}
    if kv in ("fp8", "int8"):
        dev["k_scale"] = torch.from_numpy(k_scale).to(device)
        dev["v_scale"] = torch.from_numpy(v_scale).to(device)
    return w, lens, NB, kc, vc, host, dev, alloc, sids


# --------------------------------------------------------------------------------------
# oracle timing on the host (cpu_baseline and --impl reference)
# --------------------------------------------------------------------------------------
def _oracle_task(args):
    from oracle import paged_attention
    q, kc, vc, table, t, scale = args
    t0 = time.perf_counter()
    paged_attention.paged_attention(q[None], kc, vc, table[None], np.array([t]), scale)
    return time.perf_counter() - t0


def oracle_inputs(name: str, seqs=None):
    """Per-sequence oracle inputs of the workload, built on the host with the
    oracle's own block manager and the shared generators (fp32 arrays hold the
    fp16/bf16 draws exactly)."""
    import torch
    from oracle.block_manager import BlockManager
    from paged_kv_cache_166_gb300 import workloads as W
    w = W.WORKLOADS[name]
    lens = W.context_lengths(w)
    B = w.block_size
    seqs = list(range(len(lens))) if seqs is None else seqs
    tasks = []
    for s in seqs:
        t = int(lens[s])
        nb = -(-t // B)
        # values drawn per sequence from the workload seed (the timing depends only on shapes)
        kc = W.normal_tensor((nb, w.num_kv_heads, B, w.head_dim), w.dtype, w.seed * 7919 + s,
                             W.STREAM_K_POOL).float().numpy()
        vc = W.normal_tensor((nb, w.num_kv_heads, B, w.head_dim), w.dtype, w.seed * 7919 + s,
                             W.STREAM_V_POOL).float().numpy()
        q = W.normal_tensor((w.num_q_heads, w.head_dim), w.dtype, w.seed * 7919 + s,
                            W.STREAM_Q).float().numpy()
        mgr = BlockManager(nb, B)
        sid = mgr.create()
        mgr.append(sid, t)
        table = np.asarray(mgr.tables[sid], dtype=np.int32)
        tasks.append((q, kc, vc, table, t, w.scale))
    return w, lens, seqs, tasks


def _oracle_worker(conn, name, seqs):
    """One host core: builds the oracle inputs of its sequences once, then runs the
    oracle over all of them each time the parent says go."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    _, _, _, tasks = oracle_inputs(name, seqs)
    conn.send("ready")
    while conn.recv():
        for t in tasks:
            _oracle_task(t)
        conn.send("done")
    conn.close()


def time_oracle(name: str, budget_s: float = 15.0, steps: int = 1, fill_s: float = 0.0):
    """Wall time of the oracle over a bounded sample of the workload on all host
    cores: one spawned single-threaded process per core holds its share of the
    sample (shares balanced by tokens) and runs the oracle over it on each step;
    `steps` timed passes over the same sample, each sized to about `budget_s`, and
    more passes while their total is under `fill_s` seconds."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    w, lens, _, _ = oracle_inputs(name, [])
    order = [int(s) for s in np.argsort(-lens)]  # longest first: a sample that covers the tail
    # calibrate one core on a sequence of middle length, then fill the cores: each
    # sequence (longest first) goes to the least loaded core if that core's share
    # stays within the budget; at least one sequence (the shortest)
    probe = order[len(order) // 2]
    _, _, _, tasks = oracle_inputs(name, [probe])
    per_tok = _oracle_task(tasks[0]) / max(1, int(lens[probe]))
    shares, load, sample = [[] for _ in range(cores)], [0] * cores, []
    for s in order:
        i = int(np.argmin(load))
        if (load[i] + int(lens[s])) * per_tok <= budget_s:
            shares[i].append(s)
            load[i] += int(lens[s])
            sample.append(s)
    if not sample:
        sample = [order[-1]]
        shares[0] = [order[-1]]
    ctx = mp.get_context("spawn")
    workers = []
    try:
        for sh in shares:
            if not sh:
                continue
            a, b = ctx.Pipe()
            proc = ctx.Process(target=_oracle_worker, args=(b, name, sh), daemon=True)
            proc.start()
            workers.append((proc, a))
        for _, c in workers:
            c.recv()  # inputs built
        times = []
        while len(times) < steps or sum(times) < fill_s:
            t0 = time.perf_counter()
            for _, c in workers:
                c.send(True)
            for _, c in workers:
                c.recv()
            times.append(time.perf_counter() - t0)
    finally:
        for proc, c in workers:
            try:
                c.send(False)
            except Exception:
                pass
        for proc, _ in workers:
            proc.join(timeout=10)
            if proc.is_alive():
                proc.terminate()
    elt = {"f32": 4, "f16": 2, "bf16": 2}[w.dtype]
    nbytes = attention_bytes(lens[sample], w.num_q_heads, w.num_kv_heads, w.head_dim, elt)
    return {"seconds": times, "bytes": nbytes, "tokens": int(lens[sample].sum()),
            "num_seqs": len(sample), "total_seqs": int(len(lens)), "cores": cores}


# --------------------------------------------------------------------------------------
E2E_STEPS = 48   # most timed steps of the end-to-end decode loop (contexts grow by one a step)


def measure_decode(args, name, device, rank, world, pkv, flush):
    """Times one decode workload three ways on this rank's GPU:
    * the decode step (cache write of every sequence's new token + attention), the
      bench's step, K times with CUDA events, L2 flushed between steps, clocks sampled;
    * the attention kernel alone in its own loop (the roofline figure);
    * end to end through the public API: a decode loop from the workload's state in
      which every step runs the host block manager (one new position per sequence,
      tables and lengths exported into page-locked staging memory), copies the
      step's inputs to the device in one copy, runs the decode step and reads the
      output back; contexts grow by one token a step and each step's bytes are
      counted from its own lengths.  Timed one step at a time (eager, then as a
      CUDA graph) and as a pipelined loop over two layers' caches, the host
      preparing token step i + 1 while the device runs step i."""
    import torch
    q8 = args.kv if args.kv in ("fp8", "int8") else None
    e2e_steps = max(1, min(args.steps, E2E_STEPS))
    half = max(1, e2e_steps // 2)
    # tokens every sequence gains over the three end-to-end loops (warm-up included)
    grow = 3 * (args.warmup + half) + 2
    w, lens, NB, kc, vc, host, dev, alloc, sids = build_batch(
        name, device, rank, args.kv, args.block_size, grow_tokens=grow)
    S, Hq, Hkv, D, B = len(lens), w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    elt = kc.element_size()
    q_elt = dev["q"].element_size()
    out = torch.empty_like(dev["q"])
    ws = torch.zeros(pkv.workspace_bytes(Hq, Hkv, D, q8 or dev["q"].dtype, args.num_warps),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    attn_bytes = attention_bytes(lens, Hq, Hkv, D, elt, B, q_elt)

    def decode_step(q, k_new, v_new, tables, ctx, o=None, caches=None):
        o = out if o is None else o
        kc_, vc_ = (kc, vc) if caches is None else caches
        if q8:
            fn = pkv.paged_decode_step_fp8 if q8 == "fp8" else pkv.paged_decode_step_int8
            fn(q, k_new, v_new, kc_, vc_, dev["k_scale"], dev["v_scale"], tables, ctx, w.scale,
               o, ws, args.num_warps)
        else:
            pkv.paged_decode_step(q, k_new, v_new, kc_, vc_, tables, ctx, w.scale, o, ws,
                                  args.num_warps)

    def attention(q=None, tables=None, ctx=None, o=None, caches=None):
        q = dev["q"] if q is None else q
        tables = dev["tables"] if tables is None else tables
        ctx = dev["ctx"] if ctx is None else ctx
        o = out if o is None else o
        kc_, vc_ = (kc, vc) if caches is None else caches
        if q8:
            fn = pkv.paged_decode_attention_fp8 if q8 == "fp8" else pkv.paged_decode_attention_int8
            fn(q, kc_, vc_, dev["k_scale"], dev["v_scale"], tables, ctx, w.scale, o, ws,
               args.num_warps)
        else:
            pkv.paged_decode_attention(q, kc_, vc_, tables, ctx, w.scale, o, ws, args.num_warps)

    def step():
        decode_step(dev["q"], dev["k_new"], dev["v_new"], dev["tables"], dev["ctx"])

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if pkv.decode_status(ws) != 0:
        raise RuntimeError("device status reported an error during warm-up")

    import torch.distributed as dist
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(device.index) as clocks:
        # untimed soak of the same step so that the clock samples see this load
        clocks.mark("t_soak")
        t_end = time.perf_counter() + args.soak_s
        while time.perf_counter() < t_end:
            for _ in range(20):
                flush()
                step()
            torch.cuda.synchronize()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush()              # L2 flush, outside the timed events
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
        clocks.mark("t_done")
    if world > 1:
        dist.barrier()
    ms = float(np.mean([a.elapsed_time(b) for a, b in zip(starts, ends)]))

    # the dominant kernel of a step, alone, for the roofline
    ts = []
    for i in range(args.warmup + args.steps):
        flush()
        e0.record(stream)
        attention()
        e1.record(stream)
        e1.synchronize()
        if i >= args.warmup:
            ts.append(e0.elapsed_time(e1))
    pms = float(np.mean(ts))
    status = pkv.decode_status(ws)
    if status:
        raise RuntimeError(f"device status {status} after the timed steps")

    # end to end: the decode loop through the public API (see the docstring)
    maxb = int(-(-(int(lens.max()) + grow) // B))
    names = ["q", "k_new", "v_new", "tables", "ctx"]
    sizes = {k: host[k].numel() * host[k].element_size() for k in names[:3]}
    sizes["tables"] = S * maxb * 4
    sizes["ctx"] = S * 4
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (sizes[k] + 255) & ~255
    stage_h = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    stage_d = torch.empty(total, dtype=torch.uint8, device=device)
    for k in names[:3]:
        stage_h[offs[k]:offs[k] + sizes[k]].copy_(host[k].contiguous().view(-1).view(torch.uint8))
    tab_h = stage_h[offs["tables"]:offs["tables"] + sizes["tables"]].view(torch.int32).view(S, maxb).numpy()
    ctx_h = stage_h[offs["ctx"]:offs["ctx"] + sizes["ctx"]].view(torch.int32).numpy()
    views = {}
    for k in names:
        shape = {"tables": (S, maxb), "ctx": (S,)}.get(k, tuple(host[k].shape))
        dtype = torch.int32 if k in ("tables", "ctx") else host[k].dtype
        views[k] = stage_d[offs[k]:offs[k] + sizes[k]].view(dtype).view(shape)
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    host_step = pkv.DecodeStepTables(alloc, sids, maxb, tab_h, ctx_h)

    def device_part():
        stage_d.copy_(stage_h, non_blocking=True)
        decode_step(views["q"], views["k_new"], views["v_new"], views["tables"], views["ctx"])
        out_h.copy_(out, non_blocking=True)

    def e2e_step():
        host_step()            # block manager: the step's new slots, tables into staging
        device_part()

    grown = 0

    def timed_loop(step_fn, n_warm, n_steps):
        nonlocal grown
        for _ in range(n_warm):
            flush()
            step_fn()
            grown += 1
        torch.cuda.synchronize()
        ts, nbytes = [], 0
        for _ in range(n_steps):
            flush()
            torch.cuda.synchronize()
            e0.record(stream)
            step_fn()
            e1.record(stream)
            e1.synchronize()
            grown += 1
            ts.append(e0.elapsed_time(e1))
            nbytes += attention_bytes(lens + grown, Hq, Hkv, D, elt, B, q_elt)
        return float(np.mean(ts)), nbytes / n_steps

    eager_ms, eager_bytes = timed_loop(e2e_step, args.warmup, half)
    # The same step with its copies and launches captured once in a CUDA graph and
    # replayed; the block manager still runs on the host every step and its tables
    # reach the device through the captured copy of the staging buffer.
    graph_ms = graph_bytes = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            device_part()
        torch.cuda.synchronize()

        def graph_step():
            host_step()
            g.replay()
        graph_ms, graph_bytes = timed_loop(graph_step, args.warmup, half)
    except Exception as exc:  # capture refused: report the eager loop alone
        print(f"e2e graph capture unavailable: {exc}", file=sys.stderr)
        torch.cuda.synchronize()

    # The decode loop as a server runs it, over a model of LAYERS layers: each token
    # step runs the host block manager once (one new position per sequence, tables and
    # lengths into one of two page-locked staging buffers), copies every layer's q and
    # new K/V with the tables in one H2D copy, runs the decode step on each layer's
    # cache in turn (the second cache holds the same history) and reads every layer's
    # output back.  The host prepares token step i + 1 while the device runs step i; the
    # copies go on two side streams beside the steps.  Consecutive launches read
    # different caches, so none finds the K/V of the launch before in L2 (no flush in
    # this loop); time and bytes are per layer step, all steps timed together.
    LAYERS = 2
    kc_l, vc_l = [kc, kc.clone()], [vc, vc.clone()]
    pnames = [f"{k}{l}" for l in range(LAYERS) for k in names[:3]] + ["tables", "ctx"]
    psizes = {f"{k}{l}": sizes[k] for l in range(LAYERS) for k in names[:3]}
    psizes["tables"], psizes["ctx"] = sizes["tables"], sizes["ctx"]
    poffs, ptotal = {}, 0
    for k in pnames:
        poffs[k] = ptotal
        ptotal += (psizes[k] + 255) & ~255
    stage_h2 = [torch.empty(ptotal, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    stage_d2 = [torch.empty(ptotal, dtype=torch.uint8, device=device) for _ in range(2)]
    views2, host_steps = [], []
    for b in range(2):
        for l in range(LAYERS):
            for k in names[:3]:
                o_ = poffs[f"{k}{l}"]
                stage_h2[b][o_:o_ + sizes[k]].copy_(host[k].contiguous().view(-1).view(torch.uint8))
        tab_hb = stage_h2[b][poffs["tables"]:poffs["tables"] + sizes["tables"]].view(torch.int32)
        ctx_hb = stage_h2[b][poffs["ctx"]:poffs["ctx"] + sizes["ctx"]].view(torch.int32)
        host_steps.append(pkv.DecodeStepTables(alloc, sids, maxb, tab_hb.view(S, maxb).numpy(),
                                               ctx_hb.numpy()))

        def dview(k, o_):
            v = views[k]
            return stage_d2[b][o_:o_ + sizes[k]].view(v.dtype).view(v.shape)
        tables_b, ctx_b = dview("tables", poffs["tables"]), dview("ctx", poffs["ctx"])
        views2.append([{**{k: dview(k, poffs[f"{k}{l}"]) for k in names[:3]},
                        "tables": tables_b, "ctx": ctx_b} for l in range(LAYERS)])
    out2 = [[out if (b, l) == (0, 0) else torch.empty_like(out) for l in range(LAYERS)]
            for b in range(2)]
    out_h2 = [[torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(LAYERS)]
              for _ in range(2)]
    copy_stream, back_stream = torch.cuda.Stream(device), torch.cuda.Stream(device)
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    step_done = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def layer_steps(b):
        for l in range(LAYERS):
            v = views2[b][l]
            decode_step(v["q"], v["k_new"], v["v_new"], v["tables"], v["ctx"], out2[b][l],
                        (kc_l[l], vc_l[l]))

    # a token step's launches captured once per staging buffer (eager if refused)
    step_graphs = []
    try:
        for b in (0, 1):
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2):
                layer_steps(b)
            step_graphs.append(g2)
        torch.cuda.synchronize()
    except Exception as exc:
        print(f"e2e graph capture unavailable: {exc}", file=sys.stderr)
        torch.cuda.synchronize()
        step_graphs = []

    def pipelined(n_warm, n_steps):
        nonlocal grown
        # each timed token step's bytes, counted before the loop so that the host's share
        # of a step holds only the block manager and the launches
        nbytes = LAYERS * sum(attention_bytes(lens + grown + it + 1, Hq, Hkv, D, elt, B, q_elt)
                              for it in range(n_warm, n_warm + n_steps))
        torch.cuda.synchronize()
        for it in range(n_warm + n_steps):
            if it == n_warm:
                torch.cuda.synchronize()
                e0.record(stream)
            b = it & 1
            h2d_done[b].synchronize()   # the copy of step it - 2 has read this staging buffer
            host_steps[b]()
            copy_stream.wait_event(step_done[b])  # step it - 2 is done with its device copy
            with torch.cuda.stream(copy_stream):
                stage_d2[b].copy_(stage_h2[b], non_blocking=True)
                h2d_done[b].record(copy_stream)
            stream.wait_event(h2d_done[b])
            stream.wait_event(d2h_done[b])        # step it - 2's outputs have been read back
            if step_graphs:
                step_graphs[b].replay()
            else:
                layer_steps(b)
            step_done[b].record(stream)
            back_stream.wait_event(step_done[b])
            with torch.cuda.stream(back_stream):
                for l in range(LAYERS):
                    out_h2[b][l].copy_(out2[b][l], non_blocking=True)
                d2h_done[b].record(back_stream)
            grown += 1
        stream.wait_event(d2h_done[(n_warm + n_steps - 1) & 1])  # the last read-back
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / (n_steps * LAYERS), nbytes / (n_steps * LAYERS)

    pipe_ms, pipe_bytes = pipelined(args.warmup, half)
    pipe_graph = bool(step_graphs)
    # The last layer step's read-back against the attention recomputed from its own
    # staged inputs (the cache already holds its new tokens): the same bits, or the
    # loop's buffers were reused too early.
    last = (args.warmup + half - 1) & 1
    check = torch.empty_like(out)
    v = views2[last][LAYERS - 1]
    attention(v["q"], v["tables"], v["ctx"], check, (kc_l[LAYERS - 1], vc_l[LAYERS - 1]))
    torch.cuda.synchronize()
    if not torch.equal(check.cpu().view(torch.int16), out_h2[last][LAYERS - 1].view(torch.int16)):
        raise RuntimeError("pipelined decode loop: the last read-back differs from a recomputation")
    del kc_l, vc_l
    status = pkv.decode_status(ws)
    if status:
        raise RuntimeError(f"device status {status} after the end-to-end steps")
    e2e_ms_mean, e2e_bytes_per_step = (graph_ms, graph_bytes) if graph_ms else (eager_ms, eager_bytes)
    ms, pms, e2e_ms_mean, eager_ms, pipe_ms = max_over_ranks(
        [ms, pms, e2e_ms_mean, eager_ms, pipe_ms], device)
    res = {
        "w": w, "lens": lens, "NB": NB, "q8": q8, "D": D, "bytes": attn_bytes, "ms": ms,
        "pms": pms, "e2e_ms": e2e_ms_mean, "e2e_bytes": e2e_bytes_per_step,
        "e2e_graph": graph_ms is not None, "e2e_eager_ms": eager_ms,
        "e2e_eager_bytes": eager_bytes, "e2e_pipe_ms": pipe_ms, "e2e_pipe_bytes": pipe_bytes,
        "e2e_pipe_graph": pipe_graph, "e2e_pipe_h2d": ptotal / LAYERS,
        "e2e_steps": half, "h2d": total, "d2h": out.numel() * out.element_size(),
        "clocks": clocks.summary(clocks.t_soak, clocks.t_done), "wall": wall,
        "num_warps": args.num_warps or pkv.default_num_warps(D, q8 or dev["q"].dtype),
        "q_dtype": w.dtype,
    }
    alloc.close()
    return res


def decode_record(res, world, peak, peak_kind, steps) -> dict:
    """The figures of one measured decode workload (step, kernel roofline, e2e)."""
    w, lens, q8 = res["w"], res["lens"], res["q8"]
    gbs = whole_job_gbs(res["bytes"], world, res["ms"])
    part_gbs = res["bytes"] / (res["pms"] * 1e-3) / 1e9
    tag = f"decode_attention_{q8}_{w.name}" if q8 else f"decode_attention_{w.name}"
    traffic = profile_traffic(tag)
    return {
        "value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(res["ms"], 4),
        "pct_of_peak": {"measured_copy": round(100 * gbs / peak, 1),
                        "nominal_8TBs": round(100 * gbs / NOMINAL_HBM_GBS, 1),
                        "peak_kind": peak_kind},
        "seq_tokens_per_s": round(int(lens.sum()) * world / (res["ms"] * 1e-3), 1),
        "attention_kernel": {"kv_gbs": round(part_gbs, 1), "ms": round(res["pms"], 4)},
        "roofline": {
            "bound": "hbm", "achieved": round(part_gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(part_gbs / peak, 4),
            "frac_of_nominal_8TBs": round(part_gbs / NOMINAL_HBM_GBS, 4),
            "traffic": traffic,
            "traffic_source": (f"profiles/{tag}.md (ncu dram__bytes_read.sum + "
                               "dram__bytes_write.sum of one earlier capture of the same "
                               "kernel code on this workload; not measured in this run)")
                              if traffic is not None else
                              "no ncu capture of the current kernel code on this workload",
            "kernel": "decode_attention_kernel" + (f" ({q8} cache)" if q8 else ""),
            "bytes_per_launch": res["bytes"],
            "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
        },
        "e2e": {"value": round(whole_job_gbs(res["e2e_pipe_bytes"], world, res["e2e_pipe_ms"]), 1),
                "unit": "GB/s", "ms_per_step": round(res["e2e_pipe_ms"], 4),
                "h2d_bytes_per_step": int(res["e2e_pipe_h2d"]), "d2h_bytes_per_step": int(res["d2h"]),
                "steps": res["e2e_steps"],
                "step": "one layer step of a decode loop over a two-layer model through the "
                        "public API; every token step: host block manager once "
                        "(pkv_seq_append_one_each + pkv_export_tables into one of two "
                        "page-locked staging buffers), one H2D copy of both layers' q and new "
                        "K/V with the tables and lengths (copy stream), paged_decode_step on "
                        "each layer's cache (the second a copy of the first's history), D2H of "
                        "both outputs; the host prepares token step i + 1 while the device runs "
                        "step i"
                        + ("; a token step's launches replayed from a CUDA graph per staging "
                           "buffer" if res["e2e_pipe_graph"] else "")
                        + "; copies on two side streams beside the steps; consecutive launches "
                        "read different caches (no L2 flush needed); all steps timed together "
                        "with CUDA events; contexts one token longer each token step; time, "
                        "bytes and copies per layer step",
                "sequential": {
                    "value": round(whole_job_gbs(res["e2e_bytes"], world, res["e2e_ms"]), 1),
                    "ms_per_step": round(res["e2e_ms"], 4),
                    "h2d_bytes_per_step": int(res["h2d"]),
                    "step": "one step at a time, timed alone with the L2 flushed before it: "
                            "host block manager, then the copy, the step and the read-back"
                            + ("; the copies and launches captured once in a CUDA graph and "
                               "replayed each step" if res["e2e_graph"] else "")},
                "eager": {"value": round(whole_job_gbs(res["e2e_eager_bytes"], world,
                                                       res["e2e_eager_ms"]), 1),
                          "ms_per_step": round(res["e2e_eager_ms"], 4),
                          "step": "one step at a time without the graph: every step through "
                                  "the Python API (argument checks, tensor maps, two launches, "
                                  "two copies)"}},
        "gpu_launches": 2 * steps,
        "clocks": res["clocks"],
        "wall_s_timed_loop": round(res["wall"], 3),
    }


def native(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    # the oracle pool is spawned before the first GPU call of this process
    cpu = time_oracle(args.workload, budget_s=args.cpu_budget, fill_s=args.cpu_budget) if (
        rank == 0 and world == 1 and not args.no_cpu_baseline and args.kv == "native") else None

    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_166_gb300 as pkv

    flush = L2Flush(device)
    main = measure_decode(args, args.workload, device, rank, world, pkv, flush)
    also = [] if args.also in ("", "none") else [x for x in args.also.split(",")
                                                 if x and x != args.workload]
    others = []
    for name in also:
        torch.cuda.empty_cache()   # the previous workload's caches are gone
        others.append(measure_decode(args, name, device, rank, world, pkv, flush))
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak()
    q8, w, lens = main["q8"], main["w"], main["lens"]
    rec = decode_record(main, world, peak, peak_kind, args.steps)
    line = {
        "metric": METRIC,
        "value": rec["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": f"{'e4m3' if q8 == 'fp8' else 'int8'} KV, {w.dtype} q" if q8 else w.dtype,
        "data": "synthetic",
        "config": {
            **workload_config(w, lens, main["NB"], q8),
            "step": (f"paged_decode_step_{q8}: quantising cache write of 1 new token/seq + decode "
                     "attention (2 launches, PDL-chained)") if q8 else
                    "paged_decode_step: cache write of 1 new token/seq + decode attention (2 launches, PDL-chained)",
            "l2": L2Flush.LABEL,
            "num_warps": main["num_warps"],
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
    }
    line.update({k: v for k, v in rec.items() if k not in ("value", "unit", "ms_per_step")})
    line["clocks_window"] = (f"nvidia-smi every 50 ms over a {args.soak_s} s soak of the same "
                             "step and the timed steps")
    if others:
        line["workloads"] = {}
        for o in others:
            r = decode_record(o, world, peak, peak_kind, args.steps)
            r["config"] = workload_config(o["w"], o["lens"], o["NB"], o["q8"])
            r["config"]["num_warps"] = o["num_warps"]
            line["workloads"][o["w"].name] = r
    if cpu is not None:
        cs = float(np.median(cpu["seconds"]))
        line["cpu_baseline"] = {
            "value": round(cpu["bytes"] / cs / 1e9, 4), "unit": "GB/s", "cores": cpu["cores"],
            "kind": "oracle",
            "sample": f"{cpu['num_seqs']} of {cpu['total_seqs']} sequences (longest first that fit "
                      f"the budget, {cpu['tokens']} tokens) per pass, median of "
                      f"{len(cpu['seconds'])} passes, fp64 numpy oracle, one spawned process "
                      "per core",
            "seconds": round(cs, 3)}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def kv_write_bench(args):
    """The cache write alone (pkv_kv_write): the new tokens of every sequence of the
    workload (256 for the 70B-shaped batch) scattered into the paged caches through a
    slot mapping from the library's block manager, L2 flushed between steps, CUDA
    events.  Algorithmic bytes: read k and v, write both rows, read the slots."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_166_gb300 as pkv

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w, lens, NB, kc, vc, host, dev, _, _ = build_batch(args.workload, device, 0)
    T = len(lens)
    Hkv, D = w.num_kv_heads, w.head_dim
    elt = kc.element_size()
    nbytes = kv_write_bytes(T, Hkv, D, elt)
    flush = L2Flush(device)
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def step():
        pkv.paged_kv_write(dev["k_new"], dev["v_new"], dev["slots"], kc, vc)

    ts = []
    for i in range(args.warmup + args.steps):
        flush()
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        if i >= args.warmup:
            ts.append(e0.elapsed_time(e1))
    ms = float(np.mean(ts))
    peak, peak_kind = measured_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    traffic = profile_traffic(f"kv_write_{w.name}", "kv_ops.cu")
    print(json.dumps({
        "metric": "paged_kv_write GB/s (new tokens' K/V scattered through slot_mapping)",
        "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"{w.name}: {T} new tokens, {Hkv} kv heads, head_dim {D}, "
                               f"{w.dtype}, into a pool of {NB} blocks",
                   "l2": L2Flush.LABEL},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": traffic,
                     "traffic_source": (f"profiles/kv_write_{w.name}.md (ncu dram__bytes_read.sum "
                                        "+ dram__bytes_write.sum of one earlier capture of the "
                                        "same kernel code on this workload; not measured in "
                                        "this run)") if traffic is not None else
                                       "no ncu capture of the current kernel code on this workload",
                     "kernel": "kv_write_kernel", "bytes_per_launch": nbytes,
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                     "note": "launch-bound at this size: the bytes take well under a "
                             "microsecond at the copy rate"},
        "gpu_launches": args.steps,
    }), flush=True)


def swap_bench(args):
    """Preemption by swapping: the blocks of a quarter of the workload's context
    (whole sequences, longest first) copied to page-locked host memory and back,
    timed with CUDA events; against a plain copy of the same bytes between one
    contiguous device buffer and one pinned host buffer (the link's copy rate)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_166_gb300 as pkv

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w, lens, NB, kc, vc, host, dev, _, _ = build_batch(args.workload, device, 0, args.kv)
    B = w.block_size
    nb = (lens + B - 1) // B
    tables = host["tables"].numpy()
    order = np.argsort(-lens)
    picked, total = [], 0
    for s_ in order:
        if total >= nb.sum() // 4:
            break
        picked.append(int(s_))
        total += int(nb[s_])
    ids = np.concatenate([tables[s_, :nb[s_]] for s_ in picked]).astype(np.int32)
    n = len(ids)
    ids_d = torch.from_numpy(ids).to(device)
    hk = torch.empty((n,) + tuple(kc.shape[1:]), dtype=kc.dtype).pin_memory()
    hv = torch.empty((n,) + tuple(vc.shape[1:]), dtype=vc.dtype).pin_memory()
    block_bytes = kc[0].numel() * kc.element_size()
    moved = 2 * n * block_bytes                      # K and V, one direction
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        ts = []
        for i in range(args.warmup + args.steps):
            torch.cuda.synchronize()
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if i >= args.warmup:
                ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    t_out = timed(lambda: pkv.paged_swap_out(kc, vc, ids_d, hk, hv))
    t_in = timed(lambda: pkv.paged_swap_in(hk, hv, ids_d, kc, vc))
    # the link's copy rate for the same bytes: contiguous device <-> pinned host
    dbuf = torch.empty(moved, dtype=torch.uint8, device=device)
    hbuf = torch.empty(moved, dtype=torch.uint8).pin_memory()
    c_out = timed(lambda: hbuf.copy_(dbuf, non_blocking=True))
    c_in = timed(lambda: dbuf.copy_(hbuf, non_blocking=True))
    gbs = lambda ms: moved / (ms * 1e-3) / 1e9
    value = 2 * moved / ((t_out + t_in) * 1e-3) / 1e9
    peak = 2 * moved / ((c_out + c_in) * 1e-3) / 1e9
    line = {
        "metric": "swap GB/s: a sequence set's K/V blocks to pinned host memory and back",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_out + t_in, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp8": "e4m3", "int8": "int8"}.get(args.kv, w.dtype), "data": "synthetic",
        "config": {"workload": f"{w.name}: {len(picked)} longest sequences, {n} blocks of "
                               f"{block_bytes} B per cache ({2 * n * block_bytes / 1e6:.1f} MB "
                               "each way)", "op": "paged_swap_out then paged_swap_in"},
        "swap_out": {"ms": round(t_out, 4), "gbs": round(gbs(t_out), 1)},
        "swap_in": {"ms": round(t_in, 4), "gbs": round(gbs(t_in), 1)},
        "roofline": {"bound": "link", "achieved": round(value, 1), "peak": round(peak, 1),
                     "unit": "GB/s", "frac": round(value / peak, 4), "traffic": None,
                     "peak_source": "measured in this run: contiguous cudaMemcpyAsync of the "
                                    "same bytes device->pinned host and back",
                     "copy_out_gbs": round(gbs(c_out), 1), "copy_in_gbs": round(gbs(c_in), 1)},
        "gpu_launches": 2 * args.steps,
    }
    print(json.dumps(line), flush=True)


def cow_bench(args):
    """Copy-on-write block copies in every layer's caches: one
    pkv_copy_blocks_layers launch against one pkv_copy_blocks launch per layer.
    Pairs have distinct sources and destinations (each block read once), so the
    bytes are algorithmic: read and write of K and V for every pair and layer."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_166_gb300 as pkv
    from paged_kv_cache_166_gb300 import workloads as W

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = W.WORKLOADS[args.workload]
    L, n = args.layers, args.cow_pairs
    B, Hkv, D = w.block_size, w.num_kv_heads, w.head_dim
    dt = "bf16" if w.dtype == "f32" else w.dtype
    NB = 2 * n + 16
    rng = np.random.default_rng(w.seed)
    perm = rng.permutation(NB)
    pairs = torch.from_numpy(np.stack([perm[:n], perm[n:2 * n]], 1).astype(np.int32)).to(device)
    kc = [torch.empty((NB, Hkv, B, D), dtype=W.torch_dtype(dt), device=device) for _ in range(L)]
    vc = [torch.empty_like(kc[0]) for _ in range(L)]
    for l in range(L):
        W.fill_normal_(kc[l], w.seed + l, W.STREAM_K_POOL)
        W.fill_normal_(vc[l], w.seed + l, W.STREAM_V_POOL)
    block_bytes = kc[0][0].numel() * kc[0].element_size()
    moved = 2 * 2 * L * n * block_bytes          # K and V, read and written
    flush = L2Flush(device)
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        ts = []
        for i in range(args.warmup + args.steps):
            flush()
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if i >= args.warmup:
                ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    def per_layer():
        for l in range(L):
            pkv.paged_copy_blocks(kc[l], vc[l], pairs)

    with ClockSampler(0) as clocks:
        clocks.mark("t0")
        t_one = timed(lambda: pkv.paged_copy_blocks_layers(kc, vc, pairs))
        clocks.mark("t1")
        t_per = timed(per_layer)
    gbs = lambda ms: moved / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    line = {
        "metric": "copy-on-write block copy GB/s (K and V of every layer, read + written)",
        "value": round(gbs(t_one), 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_one, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": f"{w.name} shape: {L} layers, {n} pairs with distinct source and "
                               f"destination blocks of {block_bytes} B per cache, pool {NB} blocks",
                   "op": "pkv_copy_blocks_layers (one launch)", "l2": L2Flush.LABEL},
        "per_layer_launches": {"ms": round(t_per, 4), "gbs": round(gbs(t_per), 1),
                               "launches": L},
        "roofline": {"bound": "hbm", "achieved": round(gbs(t_one), 1), "peak": peak,
                     "unit": "GB/s", "frac": round(gbs(t_one) / peak, 4), "traffic": None,
                     "kernel": "copy_blocks_layers_kernel",
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind}; copy, read + write)"},
        "clocks": clocks.summary(getattr(clocks, "t0", None), getattr(clocks, "t1", None)),
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def swap_layers_bench(args):
    """Preempting one sequence in every layer: its blocks of all L layers to pinned
    host memory and back, one launch each way, against one launch per layer and
    against a contiguous copy of the same bytes (the link's rate)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_166_gb300 as pkv
    from paged_kv_cache_166_gb300 import workloads as W

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = W.WORKLOADS[args.workload]
    L, P = args.layers, args.prefill_len
    B, Hkv, D = w.block_size, w.num_kv_heads, w.head_dim
    dt = "bf16" if w.dtype == "f32" else w.dtype
    n = -(-P // B)
    NB = 2 * n + 16
    rng = np.random.default_rng(w.seed)
    ids = torch.from_numpy(rng.permutation(NB)[:n].astype(np.int32)).to(device)
    kc = [torch.empty((NB, Hkv, B, D), dtype=W.torch_dtype(dt), device=device) for _ in range(L)]
    vc = [torch.empty_like(kc[0]) for _ in range(L)]
    for l in range(L):
        W.fill_normal_(kc[l], w.seed + l, W.STREAM_K_POOL)
        W.fill_normal_(vc[l], w.seed + l, W.STREAM_V_POOL)
    bb = kc[0][0].numel() * kc[0].element_size()
    moved = 2 * L * n * bb                        # K and V, one direction
    hk = torch.empty((L * n * bb,), dtype=torch.uint8).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        ts = []
        for i in range(args.warmup + args.steps):
            torch.cuda.synchronize()
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if i >= args.warmup:
                ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    def per_layer(out):
        for l in range(L):
            hk_l, hv_l = hk[l * n * bb:(l + 1) * n * bb], hv[l * n * bb:(l + 1) * n * bb]
            if out:
                pkv.paged_swap_out(kc[l], vc[l], ids, hk_l, hv_l)
            else:
                pkv.paged_swap_in(hk_l, hv_l, ids, kc[l], vc[l])

    t_out = timed(lambda: pkv.paged_swap_out_layers(kc, vc, ids, hk, hv))
    t_in = timed(lambda: pkv.paged_swap_in_layers(hk, hv, ids, kc, vc))
    p_out = timed(lambda: per_layer(True))
    p_in = timed(lambda: per_layer(False))
    dbuf = torch.empty(moved, dtype=torch.uint8, device=device)
    hbuf = torch.empty(moved, dtype=torch.uint8).pin_memory()
    c_out = timed(lambda: hbuf.copy_(dbuf, non_blocking=True))
    c_in = timed(lambda: dbuf.copy_(hbuf, non_blocking=True))
    gbs = lambda ms: moved / (ms * 1e-3) / 1e9
    value = 2 * moved / ((t_out + t_in) * 1e-3) / 1e9
    peak = 2 * moved / ((c_out + c_in) * 1e-3) / 1e9
    line = {
        "metric": "swap GB/s: one sequence's K/V blocks of every layer to pinned host memory "
                  "and back",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_out + t_in, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": f"{w.name} shape: {L} layers, one {P}-token sequence ({n} blocks "
                               f"of {bb} B per cache and layer, {moved / 1e6:.1f} MB each way)",
                   "op": "paged_swap_out_layers then paged_swap_in_layers (one launch each)"},
        "swap_out": {"ms": round(t_out, 4), "gbs": round(gbs(t_out), 1)},
        "swap_in": {"ms": round(t_in, 4), "gbs": round(gbs(t_in), 1)},
        "per_layer_launches": {"ms": round(p_out + p_in, 4),
                               "gbs": round(2 * moved / ((p_out + p_in) * 1e-3) / 1e9, 1),
                               "launches": 2 * L},
        "roofline": {"bound": "link", "achieved": round(value, 1), "peak": round(peak, 1),
                     "unit": "GB/s", "frac": round(value / peak, 4), "traffic": None,
                     "peak_source": "measured in this run: contiguous cudaMemcpyAsync of the "
                                    "same bytes device->pinned host and back"},
        "gpu_launches": 2 * args.steps,
    }
    print(json.dumps(line), flush=True)


def prefill_bench(args):
    """Paged prefill: every sequence's prompt processed in one causal pass (or, with
    --chunk C, its last C positions as a chunk over the rest of its context) over
    a paged cache of the workload's shape; TFLOP/s of the causal attention (4 * D
    flops per query head and visible key) against the measured bf16 tensor peak."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_166_gb300 as pkv
    from paged_kv_cache_166_gb300 import BlockAllocator
    from paged_kv_cache_166_gb300 import workloads as W

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = W.WORKLOADS[args.workload]
    dt = "bf16" if w.dtype == "f32" else w.dtype
    S, P = args.prefill_seqs, args.prefill_len
    C = args.chunk or P
    B, Hq, Hkv, D = args.block_size or w.block_size, w.num_q_heads, w.num_kv_heads, w.head_dim
    NB = S * (-(-P // B)) + 1
    alloc = BlockAllocator(NB, B, W.pool_order(NB, w.seed))
    sids = [alloc.create() for _ in range(S)]
    for s_ in sids:
        alloc.append(s_, P)
    tables, ctx = alloc.export_tables(sids, -(-P // B))
    kc = torch.empty((NB, Hkv, B, D), dtype=W.torch_dtype(dt), device=device)
    vc = torch.empty_like(kc)
    W.fill_normal_(kc, w.seed, W.STREAM_K_POOL)
    W.fill_normal_(vc, w.seed, W.STREAM_V_POOL)
    q = W.normal_tensor((S * C, Hq, D), dt, w.seed, W.STREAM_Q, device)
    out = torch.empty_like(q)
    qstart = torch.arange(0, S * C + 1, C, dtype=torch.int32, device=device)
    tab_d, ctx_d = torch.from_numpy(tables).to(device), torch.from_numpy(ctx).to(device)
    # visible keys: query i of a chunk sees P - C + i + 1 positions
    pairs = S * sum(P - C + i + 1 for i in range(C))
    flops = 4.0 * D * Hq * pairs
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush = L2Flush(device)
    step = lambda: pkv.paged_prefill_attention(q, kc, vc, tab_d, ctx_d, qstart, w.scale, out)
    ts = []
    with ClockSampler(0) as clocks:
        # untimed soak of the same launch so that the clock samples see this load
        clocks.mark("t0")
        t_end = time.perf_counter() + args.soak_s
        while time.perf_counter() < t_end:
            for _ in range(10):
                flush()
                step()
            torch.cuda.synchronize()
        for i in range(args.warmup + args.steps):
            flush()
            e0.record(stream)
            step()
            e1.record(stream)
            e1.synchronize()
            if i >= args.warmup:
                ts.append(e0.elapsed_time(e1))
        clocks.mark("t1")
    ms = float(np.median(ts))
    tflops = flops / (ms * 1e-3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        peak, kind = 1900.0, "fallback"
    line = {
        "metric": "paged prefill attention TFLOP/s (causal, 4*D flops per query head and key)",
        "value": round(tflops, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": f"{w.name} shape: {S} sequences x {P}-token context, chunk of {C} "
                               f"queries each, {Hq} q / {Hkv} kv heads, head_dim {D}, {dt}",
                   "block_size": B, "l2": L2Flush.LABEL},
        "tokens_per_s": round(S * C / (ms * 1e-3), 1),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                     "traffic": profile_traffic(f"prefill_attention_{w.name}", "prefill_tcgen05.cu",
                                                f"{w.name} {S}x{P} chunk {C}")
                     if B == w.block_size else None,
                     "kernel": "prefill_tc_kernel (tcgen05 MMAs, tensor-memory accumulators)",
                     "peak_source": f"MEASURED_PEAKS.json bf16_tflops ({kind}; dense cuBLAS)"},
        "clocks": clocks.summary(getattr(clocks, "t0", None), getattr(clocks, "t1", None)),
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def allocator_bench(args):
    """The host block manager (allocation, fork, copy-on-write, free) through the C
    ABI, on the shared-prefix parallel-sampling workload: per prompt, create and append the 1000-token prompt,
    fork the other 7 samples, then decode — one append per sample per step in round
    robin, each first write into the shared partial block a copy-on-write — until every
    sample has its suffix, and free all.  Host only, one thread; the figure includes the
    ctypes call overhead of each operation (the C++ work itself is O(1) per call)."""
    from paged_kv_cache_166_gb300 import BlockAllocator
    from paged_kv_cache_166_gb300 import workloads as W
    w = W.WORKLOADS["prefix"]
    suf = W.suffix_lengths(w)
    P, K = w.num_prompts, w.samples_per_prompt
    B = w.block_size
    blocks = P * (-(-w.prompt_len // B)) + int(sum(-(-int(x) // B) + 1 for x in suf))
    NB = int(math.ceil(blocks * (1 + w.pool_spare))) + 1

    def run():
        alloc = BlockAllocator(NB, B, W.pool_order(NB, w.seed))
        ops = cows = 0
        t0 = time.perf_counter()
        seqs = []
        for p in range(P):
            root = alloc.create()
            alloc.append(root, w.prompt_len)
            seqs.append(root)
            for _ in range(K - 1):
                seqs.append(alloc.fork(root))
            ops += 1 + 1 + (K - 1)
        left = suf.copy()
        steps = 0
        seq_ids = np.asarray(seqs, dtype=np.int32)
        while left.max() > 0:
            active = np.nonzero(left)[0]
            if args.batched:  # one call per decode step
                _, cow = alloc.append_one_each(seq_ids[active])
                cows += len(cow)
            else:
                for i in active:
                    _, cow = alloc.append(seqs[int(i)], 1)
                    cows += len(cow)
            left[active] -= 1
            ops += len(active)
            steps += 1
        for sq in seqs:
            alloc.free(sq)
            ops += 1
        dt = time.perf_counter() - t0
        assert alloc.num_free() == NB
        alloc.close()
        return ops, cows, dt, steps

    for _ in range(args.warmup):
        run()
    res = [run() for _ in range(args.steps)]
    ops, cows = res[0][0], res[0][1]
    dt = float(np.median([r[2] for r in res]))
    print(json.dumps({
        "metric": "block-manager operations per second (host, through the C ABI)",
        "value": round(ops / dt, 1), "unit": "ops/s", "n_gpus": 0, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True,
        "scaling": "none", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": f"prefix: {P} prompts x {K} samples, prompt {w.prompt_len} tokens, "
                               f"suffixes {int(suf.sum())} tokens in all, pool {NB} blocks",
                   "step": "one whole lifecycle: create + prompt append + forks, one new token "
                           "per live sample per decode step ("
                           + ("pkv_seq_append_one_each, one call per step" if args.batched
                              else "pkv_seq_append per sequence") + "), frees"},
        "ops_per_lifecycle": ops, "copy_on_write_pairs": cows,
        "us_per_op": round(dt / ops * 1e6, 3),
        "decode_steps": res[0][3],
        "gpu_launches": 0,
    }), flush=True)


REF_RUN_S = 90.0   # oracle seconds of a whole reference-arm run


def reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # every step times the same bounded sample; the sample is sized so that the
    # whole run (warm-up included) takes about REF_RUN_S seconds of oracle work
    n = args.warmup + args.steps
    per_step = min(args.ref_budget, REF_RUN_S / n)
    res = time_oracle(args.workload, budget_s=per_step, steps=n)
    times = res["seconds"][args.warmup:]
    from paged_kv_cache_166_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    sec = float(np.mean(times))
    gbs = res["bytes"] / sec / 1e9
    sample = (f"{res['num_seqs']} of {res['total_seqs']} sequences (longest first that fit the per-step budget, "
              f"{res['tokens']} tokens) per step, fp64 numpy oracle, one spawned process per core")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**workload_config(w, W.context_lengths(w), pool_blocks(w, W.context_lengths(w))),
                   "step": "fp64 numpy oracle of the decode attention on the host cores"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": res["cores"],
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="mha13b",
                    choices=["tiny", "mha13b", "gqa70b", "prefix", "longctx"])
    ap.add_argument("--num-warps", type=int, default=0)
    ap.add_argument("--also", default="gqa70b,longctx",
                    help="decode workloads timed in the same run after the main one, each "
                         "reported under 'workloads' ('none' for none)")
    ap.add_argument("--batched", type=int, default=1,
                    help="allocator bench: one batched append call per decode step (1) or one per sequence (0)")
    ap.add_argument("--op", choices=["decode", "swap", "prefill", "allocator", "cow",
                                     "swap_layers", "kv_write"],
                    default="decode",
                    help="decode: the decode step (default); swap: blocks to host and back; "
                         "prefill: causal prefill attention; allocator: the host block manager; "
                         "cow: copy-on-write block copies in every layer's caches; "
                         "kv_write: the cache write of the batch's new tokens alone; "
                         "swap_layers: one sequence (--prefill-len tokens) swapped in every "
                         "layer")
    ap.add_argument("--layers", type=int, default=32, help="layers of the cow and swap_layers ops")
    ap.add_argument("--cow-pairs", type=int, default=256, help="copy pairs of the cow op")
    ap.add_argument("--prefill-seqs", type=int, default=16)
    ap.add_argument("--prefill-len", type=int, default=2048)
    ap.add_argument("--chunk", type=int, default=0, help="prefill chunk (0: the whole prompt)")
    ap.add_argument("--block-size", type=int, default=0, choices=[0, 8, 16, 32],
                    help="cache block size (0: the workload's, 16)")
    ap.add_argument("--kv", choices=["native", "fp8", "int8"], default="native",
                    help="cache element type: the workload's dtype, or fp8 E4M3 / int8 codes "
                         "with per-KV-head scales")
    ap.add_argument("--soak-s", type=float, default=0.6,
                    help="seconds of untimed steps run just before the timed ones, so that the "
                         "clock samples cover this load")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-budget", type=float, default=5.0,
                    help="most oracle seconds of one reference-arm step (the whole run is "
                         "held to about 90 s)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.workload == "prefix":
        ap.error("the shared-prefix workload is a parity case; bench the decode batches")
    if args.op == "swap":
        swap_bench(args)
        return
    if args.op == "prefill":
        prefill_bench(args)
        return
    if args.op == "allocator":
        allocator_bench(args)
        return
    if args.op == "cow":
        cow_bench(args)
        return
    if args.op == "swap_layers":
        swap_layers_bench(args)
        return
    if args.op == "kv_write":
        kv_write_bench(args)
        return
    (reference if args.impl == "reference" else native)(args)


if __name__ == "__main__":
    main()

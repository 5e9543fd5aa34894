"""Torch-facing binding of the paged decode path: argument marshalling only.

Every function checks shapes, dtypes and devices, then calls the C ABI of
libpkv.so with raw device pointers and torch's current CUDA stream.  All the
work happens in the library's kernels; nothing here computes attention.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _native as N

_DTYPES = {torch.float32: N.PKV_F32, torch.float16: N.PKV_F16, torch.bfloat16: N.PKV_BF16}
_CODES = {"fp8": N.PKV_FP8_E4M3, "int8": N.PKV_INT8}   # the 8-bit cache kinds
_WORKSPACES: dict = {}


def dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check_cuda(*ts) -> torch.device:
    dev = ts[0].device
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")
        if t.device != dev:
            raise ValueError("tensors must be on one device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    return dev


def _check_index(t: torch.Tensor, name: str) -> None:
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")


def paged_kv_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    """Scatter k, v [T, Hkv, D] into k_cache, v_cache [NB, Hkv, B, D] at slot_mapping [T]."""
    dev = _check_cuda(k, v, slot_mapping, k_cache, v_cache)
    _check_index(slot_mapping, "slot_mapping")
    if k.shape != v.shape or k_cache.shape != v_cache.shape or k.dim() != 3 or k_cache.dim() != 4:
        raise ValueError("expected k, v [T, Hkv, D] and caches [NB, Hkv, B, D]")
    T, Hkv, D = k.shape
    NB, Hkv2, B, D2 = k_cache.shape
    if (Hkv, D) != (Hkv2, D2) or slot_mapping.shape != (T,):
        raise ValueError("shape mismatch between tokens, slots and caches")
    if not (k.dtype == v.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("k, v and caches must share a dtype")
    N.check(N.lib().pkv_kv_write(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
                                 k_cache.data_ptr(), v_cache.data_ptr(), NB, Hkv, B, D,
                                 dtype_code(k), _stream(dev)))


def default_num_warps(head_dim: int, dtype) -> int:
    """Default worker warps; ``dtype`` as in ``workspace_bytes``."""
    code = _CODES[dtype] if isinstance(dtype, str) else _DTYPES[dtype]
    n = ctypes.c_int32(0)
    N.check(N.lib().pkv_decode_default_warps(head_dim, code, ctypes.byref(n)))
    return n.value


def workspace_bytes(num_q_heads: int, num_kv_heads: int, head_dim: int, dtype,
                    num_warps: int = 0) -> int:
    """Decode workspace bytes; ``dtype`` is q's torch dtype, or "fp8" / "int8"
    for attention over that 8-bit cache."""
    code = _CODES[dtype] if isinstance(dtype, str) else _DTYPES[dtype]
    n = ctypes.c_size_t(0)
    N.check(N.lib().pkv_decode_workspace_size(num_q_heads, num_kv_heads, head_dim, code,
                                              num_warps, ctypes.byref(n)))
    return n.value


def get_workspace(device: torch.device, group: int, head_dim: int, num_warps: int,
                  nbytes: int, kind: str = "") -> torch.Tensor:
    """A zero-filled device workspace of ``nbytes`` for one layout (group size,
    head_dim, warp count, cache kind), cached per device and stream: one workspace
    must not serve two launches that may overlap, nor two layouts."""
    key = (device.index, torch.cuda.current_stream(device).cuda_stream, group, head_dim,
           num_warps, kind)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _WORKSPACES[key] = ws
    return ws


def _decode_shapes(q, k_cache, v_cache, block_tables, context_lens, out):
    if q.dim() != 3 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("expected q [S, Hq, D] and caches [NB, Hkv, B, D]")
    S, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    if D2 != D or out.shape != q.shape:
        raise ValueError("head_dim mismatch or out shape != q shape")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks] and context_lens [S]")
    if not (q.dtype == k_cache.dtype == v_cache.dtype == out.dtype):
        raise TypeError("q, caches and out must share a dtype")
    _check_index(block_tables, "block_tables")
    _check_index(context_lens, "context_lens")
    return S, Hq, D, NB, Hkv, B, block_tables.shape[1]


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           out: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                           num_warps: int = 0) -> torch.Tensor:
    """Decode attention of q [S, Hq, D] over the paged caches; writes and returns out."""
    dev = _check_cuda(q, k_cache, v_cache, block_tables, context_lens, out)
    S, Hq, D, NB, Hkv, B, MAXB = _decode_shapes(q, k_cache, v_cache, block_tables,
                                                context_lens, out)
    need = workspace_bytes(Hq, Hkv, D, q.dtype, num_warps)
    ws = get_workspace(dev, Hq // Hkv, D, num_warps, need) if workspace is None else workspace
    if ws.numel() * ws.element_size() < need:
        raise ValueError(f"workspace smaller than the {need} bytes needed")
    N.check(N.lib().pkv_decode_attention(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), MAXB,
        context_lens.data_ptr(), S, Hq, Hkv, D, B, NB, float(scale), out.data_ptr(),
        ws.data_ptr(), ws.numel() * ws.element_size(), num_warps, dtype_code(q), _stream(dev)))
    return out


def paged_decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                      workspace: Optional[torch.Tensor] = None, num_warps: int = 0) -> torch.Tensor:
    """One decode step: write each sequence's new token (k_new, v_new [S, Hkv, D],
    position context_lens[s] - 1, slot from the block table) into the caches, then
    attend over them (two launches chained with programmatic dependent launch)."""
    dev = _check_cuda(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out)
    S, Hq, D, NB, Hkv, B, MAXB = _decode_shapes(q, k_cache, v_cache, block_tables,
                                                context_lens, out)
    if k_new.shape != (S, Hkv, D) or v_new.shape != (S, Hkv, D):
        raise ValueError("k_new and v_new must be [S, Hkv, D]")
    if k_new.dtype != q.dtype or v_new.dtype != q.dtype:
        raise TypeError("k_new and v_new must share the dtype of q")
    need = workspace_bytes(Hq, Hkv, D, q.dtype, num_warps)
    ws = get_workspace(dev, Hq // Hkv, D, num_warps, need) if workspace is None else workspace
    if ws.numel() * ws.element_size() < need:
        raise ValueError(f"workspace smaller than the {need} bytes needed")
    N.check(N.lib().pkv_decode_step(
        q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), MAXB, context_lens.data_ptr(), S, Hq, Hkv, D, B, NB,
        float(scale), out.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(), num_warps,
        dtype_code(q), _stream(dev)))
    return out


def _q8_caches(k_cache, v_cache, kind):
    """(k_cache, v_cache) as byte views: fp8 caches are uint8 or float8_e4m3fn
    tensors, int8 caches int8 tensors."""
    out = []
    for c in (k_cache, v_cache):
        if kind == "fp8":
            if c.dtype == getattr(torch, "float8_e4m3fn", None):
                c = c.view(torch.uint8)
            if c.dtype != torch.uint8:
                raise TypeError("fp8 caches must be uint8 or float8_e4m3fn tensors")
        elif c.dtype != torch.int8:
            raise TypeError("int8 caches must be int8 tensors")
        out.append(c)
    return out


def _check_scales(k_scale, v_scale, Hkv):
    for t in (k_scale, v_scale):
        if t.dtype != torch.float32 or t.shape != (Hkv,):
            raise ValueError(f"scales must be float32 [{Hkv}]")


def _kv_write_q8(kind, k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale):
    kc, vc = _q8_caches(k_cache, v_cache, kind)
    dev = _check_cuda(k, v, slot_mapping, kc, vc, k_scale, v_scale)
    _check_index(slot_mapping, "slot_mapping")
    if k.shape != v.shape or k.dim() != 3 or kc.dim() != 4 or vc.dim() != 4:
        raise ValueError("expected k, v [T, Hkv, D], k_cache [NB, Hkv, 16, D], v_cache [NB, Hkv, D, 16]")
    T, Hkv, D = k.shape
    NB, B = kc.shape[0], kc.shape[2]
    if kc.shape != (NB, Hkv, B, D) or vc.shape != (NB, Hkv, D, B) or slot_mapping.shape != (T,):
        raise ValueError(f"shape mismatch between tokens, slots and {kind} caches")
    _check_scales(k_scale, v_scale, Hkv)
    if k.dtype != v.dtype:
        raise TypeError("k and v must share a dtype")
    fn = N.lib().pkv_kv_write_fp8 if kind == "fp8" else N.lib().pkv_kv_write_int8
    N.check(fn(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T, kc.data_ptr(),
               vc.data_ptr(), k_scale.data_ptr(), v_scale.data_ptr(), NB, Hkv, B, D,
               dtype_code(k), _stream(dev)))


def paged_kv_write_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                       k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                       v_scale: torch.Tensor) -> None:
    """Quantise k, v [T, Hkv, D] to fp8 (E4M3, per-KV-head scales) and scatter them:
    k_cache [NB, Hkv, 16, D], v_cache [NB, Hkv, D, 16] (uint8)."""
    _kv_write_q8("fp8", k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale)


def paged_kv_write_int8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                        k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                        v_scale: torch.Tensor) -> None:
    """Quantise k, v [T, Hkv, D] to int8 codes in [-127, 127] (per-KV-head scales)
    and scatter them: k_cache [NB, Hkv, 16, D], v_cache [NB, Hkv, D, 16] (int8)."""
    _kv_write_q8("int8", k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale)


def _q8_shapes(q, kc, vc, block_tables, context_lens, out):
    if q.dim() != 3 or kc.dim() != 4 or vc.dim() != 4:
        raise ValueError("expected q [S, Hq, D], k_cache [NB, Hkv, 16, D], v_cache [NB, Hkv, D, 16]")
    S, Hq, D = q.shape
    NB, Hkv, B, D2 = kc.shape
    if D2 != D or vc.shape != (NB, Hkv, D, B) or out.shape != q.shape:
        raise ValueError("head_dim mismatch, v_cache not [NB, Hkv, D, 16] or out shape != q shape")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks] and context_lens [S]")
    if q.dtype != out.dtype:
        raise TypeError("q and out must share a dtype")
    _check_index(block_tables, "block_tables")
    _check_index(context_lens, "context_lens")
    return S, Hq, D, NB, Hkv, B, block_tables.shape[1]


def _q8_workspace(kind, dev, Hq, Hkv, D, num_warps, workspace):
    need = workspace_bytes(Hq, Hkv, D, kind, num_warps)
    ws = get_workspace(dev, Hq // Hkv, D, num_warps, need, kind) if workspace is None else workspace
    if ws.numel() * ws.element_size() < need:
        raise ValueError(f"workspace smaller than the {need} bytes needed")
    return ws


def _decode_attention_q8(kind, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                         context_lens, scale, out, workspace, num_warps):
    kc, vc = _q8_caches(k_cache, v_cache, kind)
    dev = _check_cuda(q, kc, vc, k_scale, v_scale, block_tables, context_lens, out)
    S, Hq, D, NB, Hkv, B, MAXB = _q8_shapes(q, kc, vc, block_tables, context_lens, out)
    _check_scales(k_scale, v_scale, Hkv)
    ws = _q8_workspace(kind, dev, Hq, Hkv, D, num_warps, workspace)
    fn = N.lib().pkv_decode_attention_fp8 if kind == "fp8" else N.lib().pkv_decode_attention_int8
    N.check(fn(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), k_scale.data_ptr(), v_scale.data_ptr(),
               block_tables.data_ptr(), MAXB, context_lens.data_ptr(), S, Hq, Hkv, D, B, NB,
               float(scale), out.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(),
               num_warps, dtype_code(q), _stream(dev)))
    return out


def _decode_step_q8(kind, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables,
                    context_lens, scale, out, workspace, num_warps):
    kc, vc = _q8_caches(k_cache, v_cache, kind)
    dev = _check_cuda(q, k_new, v_new, kc, vc, k_scale, v_scale, block_tables, context_lens, out)
    S, Hq, D, NB, Hkv, B, MAXB = _q8_shapes(q, kc, vc, block_tables, context_lens, out)
    _check_scales(k_scale, v_scale, Hkv)
    if k_new.shape != (S, Hkv, D) or v_new.shape != (S, Hkv, D):
        raise ValueError("k_new and v_new must be [S, Hkv, D]")
    if k_new.dtype != q.dtype or v_new.dtype != q.dtype:
        raise TypeError("k_new and v_new must share the dtype of q")
    ws = _q8_workspace(kind, dev, Hq, Hkv, D, num_warps, workspace)
    fn = N.lib().pkv_decode_step_fp8 if kind == "fp8" else N.lib().pkv_decode_step_int8
    N.check(fn(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), kc.data_ptr(), vc.data_ptr(),
               k_scale.data_ptr(), v_scale.data_ptr(), block_tables.data_ptr(), MAXB,
               context_lens.data_ptr(), S, Hq, Hkv, D, B, NB, float(scale), out.data_ptr(),
               ws.data_ptr(), ws.numel() * ws.element_size(), num_warps, dtype_code(q),
               _stream(dev)))
    return out


def paged_decode_attention_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               k_scale: torch.Tensor, v_scale: torch.Tensor,
                               block_tables: torch.Tensor, context_lens: torch.Tensor,
                               scale: float, out: torch.Tensor,
                               workspace: Optional[torch.Tensor] = None,
                               num_warps: int = 0) -> torch.Tensor:
    """Decode attention of q [S, Hq, D] (f16/bf16) over fp8 caches; writes and returns out."""
    return _decode_attention_q8("fp8", q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                context_lens, scale, out, workspace, num_warps)


def paged_decode_attention_int8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                k_scale: torch.Tensor, v_scale: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor,
                                scale: float, out: torch.Tensor,
                                workspace: Optional[torch.Tensor] = None,
                                num_warps: int = 0) -> torch.Tensor:
    """Decode attention of q [S, Hq, D] (f16/bf16) over int8 caches; writes and returns out."""
    return _decode_attention_q8("int8", q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                context_lens, scale, out, workspace, num_warps)


def paged_decode_step_fp8(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                          k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                          v_scale: torch.Tensor, block_tables: torch.Tensor,
                          context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                          workspace: Optional[torch.Tensor] = None,
                          num_warps: int = 0) -> torch.Tensor:
    """One decode step over fp8 caches: quantise and write each sequence's new token
    (position context_lens[s] - 1), then attend (two launches, programmatic
    dependent launch)."""
    return _decode_step_q8("fp8", q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                           block_tables, context_lens, scale, out, workspace, num_warps)


def paged_decode_step_int8(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                           k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                           v_scale: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                           workspace: Optional[torch.Tensor] = None,
                           num_warps: int = 0) -> torch.Tensor:
    """One decode step over int8 caches: quantise and write each sequence's new
    token (position context_lens[s] - 1), then attend (two launches, programmatic
    dependent launch)."""
    return _decode_step_q8("int8", q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                           block_tables, context_lens, scale, out, workspace, num_warps)


def paged_prefill_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor,
                            query_start: torch.Tensor, scale: float, out: torch.Tensor,
                            status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Causal attention of each sequence's chunk of queries q [T, Hq, D] (rows
    query_start[s]..query_start[s+1]-1, the last positions of context_lens[s]) over
    the paged caches; writes and returns out."""
    dev = _check_cuda(q, k_cache, v_cache, block_tables, context_lens, query_start, out)
    if q.dim() != 3 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape or out.shape != q.shape:
        raise ValueError("expected q, out [T, Hq, D] and caches [NB, Hkv, B, D]")
    T, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    S = context_lens.shape[0]
    if D2 != D or block_tables.dim() != 2 or block_tables.shape[0] != S or query_start.shape != (S + 1,):
        raise ValueError("block_tables [S, max_blocks], context_lens [S], query_start [S + 1]")
    for t, n in ((block_tables, "block_tables"), (context_lens, "context_lens"),
                 (query_start, "query_start")):
        _check_index(t, n)
    if not (q.dtype == k_cache.dtype == v_cache.dtype == out.dtype):
        raise TypeError("q, caches and out must share a dtype")
    st = 0
    if status is not None:
        _check_cuda(status)
        if status.dtype != torch.int32 or status.numel() < 1:
            raise ValueError("status must be a device int32 tensor")
        st = status.data_ptr()
    N.check(N.lib().pkv_prefill_attention(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), query_start.data_ptr(), S, T, Hq, Hkv, D, B,
        NB, float(scale), out.data_ptr(), st or None, dtype_code(q), _stream(dev)))
    return out


def _swap_args(k_cache, v_cache, block_ids, host_k, host_v):
    dev = _check_cuda(k_cache, v_cache, block_ids)
    _check_index(block_ids, "block_ids")
    if block_ids.dim() != 1:
        raise ValueError("block_ids must be [n]")
    n = block_ids.shape[0]
    block_bytes = k_cache[0].numel() * k_cache.element_size()
    if v_cache.shape[0] != k_cache.shape[0] or v_cache[0].numel() * v_cache.element_size() != block_bytes:
        raise ValueError("K and V caches must hold blocks of the same size")
    for h in (host_k, host_v):
        if h.is_cuda or not h.is_pinned() or not h.is_contiguous():
            raise ValueError("host buffers must be contiguous page-locked (pinned) CPU tensors")
        if h.numel() * h.element_size() < n * block_bytes:
            raise ValueError(f"host buffer smaller than {n} blocks of {block_bytes} bytes")
    return dev, n, block_bytes


def paged_swap_out(k_cache: torch.Tensor, v_cache: torch.Tensor, block_ids: torch.Tensor,
                   host_k: torch.Tensor, host_v: torch.Tensor) -> None:
    """Copy cache blocks block_ids (device int32 [n]) to pinned host buffers: host
    block i = cache block block_ids[i], K and V."""
    dev, n, bb = _swap_args(k_cache, v_cache, block_ids, host_k, host_v)
    N.check(N.lib().pkv_swap_out_blocks(k_cache.data_ptr(), v_cache.data_ptr(),
                                        block_ids.data_ptr(), n, k_cache.shape[0], bb,
                                        host_k.data_ptr(), host_v.data_ptr(), _stream(dev)))


def paged_swap_in(host_k: torch.Tensor, host_v: torch.Tensor, block_ids: torch.Tensor,
                  k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    """Copy pinned host blocks back: cache block block_ids[i] = host block i."""
    dev, n, bb = _swap_args(k_cache, v_cache, block_ids, host_k, host_v)
    N.check(N.lib().pkv_swap_in_blocks(host_k.data_ptr(), host_v.data_ptr(),
                                       block_ids.data_ptr(), n, k_cache.shape[0], bb,
                                       k_cache.data_ptr(), v_cache.data_ptr(), _stream(dev)))


def _swap_layers_args(k_caches, v_caches, block_ids, host_k, host_v):
    k_caches, v_caches = list(k_caches), list(v_caches)
    if not k_caches or len(k_caches) != len(v_caches):
        raise ValueError("one K and one V cache per layer, at least one layer")
    ref = k_caches[0]
    for c in k_caches + v_caches:
        if c.shape != ref.shape or c.element_size() != ref.element_size():
            raise ValueError("every layer's caches must hold blocks of one shape")
    dev = _check_cuda(*k_caches, *v_caches, block_ids)
    _check_index(block_ids, "block_ids")
    if block_ids.dim() != 1:
        raise ValueError("block_ids must be [n]")
    L, n = len(k_caches), block_ids.shape[0]
    block_bytes = ref[0].numel() * ref.element_size()
    for h in (host_k, host_v):
        if h.is_cuda or not h.is_pinned() or not h.is_contiguous():
            raise ValueError("host buffers must be contiguous page-locked (pinned) CPU tensors")
        if h.numel() * h.element_size() < L * n * block_bytes:
            raise ValueError(f"host buffer smaller than {L} layers x {n} blocks of "
                             f"{block_bytes} bytes")
    kp = (ctypes.c_void_p * L)(*[c.data_ptr() for c in k_caches])
    vp = (ctypes.c_void_p * L)(*[c.data_ptr() for c in v_caches])
    return dev, L, n, ref.shape[0], block_bytes, kp, vp


def paged_swap_out_layers(k_caches, v_caches, block_ids: torch.Tensor, host_k: torch.Tensor,
                          host_v: torch.Tensor) -> None:
    """paged_swap_out for every layer's caches in one launch: layer l's copy of
    block block_ids[i] goes to host block l * n + i (host buffers of L * n blocks)."""
    dev, L, n, NB, bb, kp, vp = _swap_layers_args(k_caches, v_caches, block_ids, host_k, host_v)
    N.check(N.lib().pkv_swap_out_blocks_layers(kp, vp, L, block_ids.data_ptr(), n, NB, bb,
                                               host_k.data_ptr(), host_v.data_ptr(),
                                               _stream(dev)))


def paged_swap_in_layers(host_k: torch.Tensor, host_v: torch.Tensor, block_ids: torch.Tensor,
                         k_caches, v_caches) -> None:
    """paged_swap_in for every layer's caches in one launch: layer l's block
    block_ids[i] = host block l * n + i."""
    dev, L, n, NB, bb, kp, vp = _swap_layers_args(k_caches, v_caches, block_ids, host_k, host_v)
    N.check(N.lib().pkv_swap_in_blocks_layers(host_k.data_ptr(), host_v.data_ptr(),
                                              block_ids.data_ptr(), n, NB, bb, kp, vp, L,
                                              _stream(dev)))


def decode_status(workspace: torch.Tensor) -> int:
    """Reads and clears the device status bits the decode kernels recorded."""
    v = ctypes.c_int32(0)
    N.check(N.lib().pkv_decode_status(workspace.data_ptr(), ctypes.byref(v),
                                      _stream(workspace.device)))
    return v.value


def wait_timeout_selftest(limit_us: int = 20000, device=None) -> tuple:
    """Runs the library's bounded-wait self-test on ``device`` (default: the current
    CUDA device) and returns (status bits, nanoseconds the first wait lasted, whether
    the wait after completing the barrier succeeded).  A healthy device gives
    (PKV_DEV_WAIT_TIMEOUT, >= limit_us * 1000, True)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    report = torch.zeros(2, dtype=torch.int64, device=dev)
    N.check(N.lib().pkv_wait_timeout_selftest(status.data_ptr(), report.data_ptr(), int(limit_us),
                                              _stream(dev)))
    r = report.cpu()
    return int(status.item()), int(r[0]), bool(r[1] == 1)


def _copy_code(cache: torch.Tensor) -> int:
    if cache.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        return N.PKV_FP8_E4M3
    if cache.dtype == torch.int8:
        return N.PKV_INT8
    return dtype_code(cache)


def paged_copy_blocks_layers(k_caches, v_caches, src_dst_pairs: torch.Tensor) -> None:
    """Copy whole blocks src -> dst in every layer's K and V caches, one launch
    (lists of per-layer caches of one shape; pairs [n, 2] int32 on their device)."""
    k_caches, v_caches = list(k_caches), list(v_caches)
    if not k_caches or len(k_caches) != len(v_caches):
        raise ValueError("one K and one V cache per layer, at least one layer")
    dev = _check_cuda(*k_caches, *v_caches, src_dst_pairs)
    _check_index(src_dst_pairs, "src_dst_pairs")
    n = src_dst_pairs.numel() // 2
    if src_dst_pairs.numel() != 2 * n:
        raise ValueError("src_dst_pairs must hold pairs")
    ref = k_caches[0]
    for c in k_caches + v_caches:
        if c.shape != ref.shape or c.dtype != ref.dtype:
            raise ValueError("every layer's caches must have one shape and dtype")
    L = len(k_caches)
    kp = (ctypes.c_void_p * L)(*[c.data_ptr() for c in k_caches])
    vp = (ctypes.c_void_p * L)(*[c.data_ptr() for c in v_caches])
    N.check(N.lib().pkv_copy_blocks_layers(kp, vp, L, src_dst_pairs.data_ptr(), n, ref.shape[0],
                                           ref[0].numel(), _copy_code(ref), _stream(dev)))


def paged_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor,
                      src_dst_pairs: torch.Tensor) -> None:
    """Copy whole blocks src -> dst (pairs [n, 2] int32 on the caches' device)."""
    dev = _check_cuda(k_cache, v_cache, src_dst_pairs)
    _check_index(src_dst_pairs, "src_dst_pairs")
    n = src_dst_pairs.numel() // 2
    if src_dst_pairs.numel() != 2 * n:
        raise ValueError("src_dst_pairs must hold pairs")
    NB = k_cache.shape[0]
    block_elems = k_cache[0].numel()
    if k_cache.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        code = N.PKV_FP8_E4M3
    elif k_cache.dtype == torch.int8:
        code = N.PKV_INT8
    else:
        code = dtype_code(k_cache)
    N.check(N.lib().pkv_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(),
                                    src_dst_pairs.data_ptr(), n, NB, block_elems, code,
                                    _stream(dev)))

"""ctypes declarations of libpkv.so (the C ABI in include/pkv.h).

The library is loaded lazily on first use.  If it has not been built, every
call raises: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_DTYPE = -2
PKV_ERR_OUT_OF_BLOCKS = -3
PKV_ERR_CUDA = -4
PKV_ERR_UNSUPPORTED = -5
PKV_ERR_DEVICE = -6

PKV_F32, PKV_F16, PKV_BF16, PKV_FP8_E4M3, PKV_INT8 = 0, 1, 2, 3, 4

PKV_DEV_BAD_CONTEXT_LEN = 1
PKV_DEV_BAD_BLOCK_ID = 2
PKV_DEV_WAIT_TIMEOUT = 4
PKV_DEV_WORKSPACE_MISMATCH = 8

PKV_STATIC_SCRATCH_BYTES = 16 << 20

_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_p = ctypes.c_void_p
_pi32 = ctypes.POINTER(ctypes.c_int32)
_sz = ctypes.c_size_t
_f = ctypes.c_float

SIGNATURES = {
    "pkv_last_error_string": (ctypes.c_char_p, []),
    "pkv_version": (ctypes.c_int, []),
    "pkv_wait_timeout_selftest": (ctypes.c_int, [_p, _p, _i32, _p]),
    "pkv_kv_write": (ctypes.c_int, [_p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32, _i32, _p]),
    "pkv_decode_workspace_size": (ctypes.c_int, [_i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_sz)]),
    "pkv_decode_attention": (ctypes.c_int, [_p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32,
                                            _i32, _f, _p, _p, _sz, _i32, _i32, _p]),
    "pkv_decode_step": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32,
                                       _i32, _i32, _f, _p, _p, _sz, _i32, _i32, _p]),
    "pkv_decode_status": (ctypes.c_int, [_p, _pi32, _p]),
    "pkv_decode_default_warps": (ctypes.c_int, [_i32, _i32, _pi32]),
    "pkv_decode_attention_static_scratch": (ctypes.c_int, [_p, _p, _p, _p, _i32, _p, _i32, _i32,
                                                           _i32, _i32, _i32, _i32, _f, _p, _i32,
                                                           _i32, _p]),
    "pkv_copy_blocks": (ctypes.c_int, [_p, _p, _p, _i32, _i32, _i64, _i32, _p]),
    "pkv_copy_blocks_layers": (ctypes.c_int, [_p, _p, _i32, _p, _i32, _i32, _i64, _i32, _p]),
    "pkv_prefill_attention": (ctypes.c_int, [_p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32,
                                             _i32, _i32, _i32, _f, _p, _p, _i32, _p]),
    "pkv_swap_out_blocks": (ctypes.c_int, [_p, _p, _p, _i32, _i32, _i64, _p, _p, _p]),
    "pkv_swap_in_blocks": (ctypes.c_int, [_p, _p, _p, _i32, _i32, _i64, _p, _p, _p]),
    "pkv_swap_out_blocks_layers": (ctypes.c_int, [_p, _p, _i32, _p, _i32, _i32, _i64, _p, _p,
                                                  _p]),
    "pkv_swap_in_blocks_layers": (ctypes.c_int, [_p, _p, _p, _i32, _i32, _i64, _p, _p, _i32,
                                                 _p]),
    "pkv_seq_swap_out": (ctypes.c_int, [_p, _i32, _pi32, _i32, _pi32]),
    "pkv_seq_swap_in": (ctypes.c_int, [_p, _i32, _pi32, _i32, _pi32]),
    "pkv_kv_write_fp8": (ctypes.c_int, [_p, _p, _p, _i32, _p, _p, _p, _p, _i32, _i32, _i32, _i32,
                                        _i32, _p]),
    "pkv_decode_attention_fp8": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _i32,
                                                _i32, _i32, _i32, _f, _p, _p, _sz, _i32, _i32,
                                                _p]),
    "pkv_decode_step_fp8": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32,
                                           _i32, _i32, _i32, _i32, _f, _p, _p, _sz, _i32, _i32,
                                           _p]),
    "pkv_kv_write_int8": (ctypes.c_int, [_p, _p, _p, _i32, _p, _p, _p, _p, _i32, _i32, _i32, _i32,
                                         _i32, _p]),
    "pkv_decode_attention_int8": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32,
                                                 _i32, _i32, _i32, _i32, _f, _p, _p, _sz, _i32,
                                                 _i32, _p]),
    "pkv_decode_step_int8": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32,
                                            _i32, _i32, _i32, _i32, _f, _p, _p, _sz, _i32, _i32,
                                            _p]),
    "pkv_allocator_create": (ctypes.c_int, [_i32, _i32, _pi32, ctypes.POINTER(_p)]),
    "pkv_allocator_destroy": (ctypes.c_int, [_p]),
    "pkv_block_alloc": (ctypes.c_int, [_p, _pi32]),
    "pkv_block_incref": (ctypes.c_int, [_p, _i32]),
    "pkv_block_decref": (ctypes.c_int, [_p, _i32]),
    "pkv_block_refcount": (ctypes.c_int, [_p, _i32, _pi32]),
    "pkv_num_free_blocks": (ctypes.c_int, [_p, _pi32]),
    "pkv_seq_create": (ctypes.c_int, [_p, _pi32]),
    "pkv_seq_fork": (ctypes.c_int, [_p, _i32, _pi32]),
    "pkv_seq_free": (ctypes.c_int, [_p, _i32]),
    "pkv_seq_blocks_needed": (ctypes.c_int, [_p, _i32, _i32, _pi32]),
    "pkv_seq_append": (ctypes.c_int, [_p, _i32, _i32, _pi32, _pi32, _pi32]),
    "pkv_seq_append_one_each": (ctypes.c_int, [_p, _pi32, _i32, _pi32, _pi32, _pi32]),
    "pkv_seq_len": (ctypes.c_int, [_p, _i32, _pi32]),
    "pkv_seq_table": (ctypes.c_int, [_p, _i32, _pi32, _i32, _pi32]),
    "pkv_export_tables": (ctypes.c_int, [_p, _pi32, _i32, _i32, _pi32, _pi32]),
}

_lib = None
_lock = threading.Lock()


class PkvError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"pkv error {code}: {message}")
        self.code = code


class OutOfBlocks(PkvError):
    pass


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; "
                        f"g.build()\"` (or paged_kv_cache_166_gb300/build.py)")
                L = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(L, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = L
    return _lib


def check(code: int) -> None:
    if code != PKV_OK:
        msg = lib().pkv_last_error_string().decode(errors="replace")
        if code == PKV_ERR_OUT_OF_BLOCKS:
            raise OutOfBlocks(code, msg)
        raise PkvError(code, msg)

"""Python binding of the quantized K/V cache library (include/kvq.h).

Thin ctypes marshalling over libkvq.so: every function has the name of the C
entry point it calls and only converts arguments (torch tensors -> device
pointers, the current torch CUDA stream -> cudaStream_t).  All work happens
in the library's CUDA kernels; there is no fallback of any kind.  If the
library has not been built, importing the binding's functions raises.

    from quantized_kv_cache_append_gb300 import (
        KVQ_F16, KVQ_Q8, kvq_cache, kvq_append, kvq_decode_attn, ...)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from .build import LIB_PATH, build  # noqa: F401  (build() is the in-tree nvcc build)

KVQ_F16 = 0
KVQ_Q8 = 1
KVQ_K8V4 = 2
KVQ_GROUP = 64
KVQ_Q4_BLOCK = 32

KVQ_OK = 0
KVQ_ERR_ARG = 1
KVQ_ERR_UNSUPPORTED = 2
KVQ_ERR_WORKSPACE = 3
KVQ_ERR_CUDA = 4

# Every symbol the C header declares, in the order it declares them.
EXPORTED_SYMBOLS = (
    "kvq_block_bytes",
    "kvq_append",
    "kvq_decode_workspace_bytes",
    "kvq_decode_attn",
    "kvq_decode_attn_lost_wait_test",
    "kvq_compact_f16",
    "kvq_chunk_attn",
    "kvq_chunk_attn_lost_wait_test",
    "kvq_gather_cells",
    "kvq_scatter_cells",
    "kvq_stream_plan",
    "kvq_stream_fetch",
    "kvq_decode_attn_static",
    "kvq_status_string",
)

# Size of the library-held scratch used by kvq_decode_attn_static.
KVQ_STATIC_SCRATCH_BYTES = 8 << 20


class kvq_cache(ctypes.Structure):
    """Mirror of `struct kvq_cache` (one layer's paged pool descriptor)."""

    _fields_ = [
        ("fmt", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("n_blocks", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("k_data", ctypes.c_void_p),
        ("v_data", ctypes.c_void_p),
        ("k_scales", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
    ]


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {kvq_status_string(status)}")
        self.status = status


_lib = None


def load_library(path: Optional[str] = None):
    """Load libkvq.so (raises if it is missing: there is no other path)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library not built: {p} is missing "
            "(run quantized_kv_cache_append_gb300.build.build())")
    lib = ctypes.CDLL(p)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    CP = ctypes.POINTER(kvq_cache)
    lib.kvq_block_bytes.restype = Z
    lib.kvq_block_bytes.argtypes = [I, I, I, I]
    lib.kvq_append.restype = I
    lib.kvq_append.argtypes = [CP, P, P, I, P, P, P, I, I, P]
    lib.kvq_decode_workspace_bytes.restype = Z
    lib.kvq_decode_workspace_bytes.argtypes = [CP, I, I, I, I]
    lib.kvq_decode_attn.restype = I
    lib.kvq_decode_attn.argtypes = [CP, P, I, I, I, P, I, P, I, ctypes.c_float, P, P, Z, P]
    lib.kvq_decode_attn_lost_wait_test.restype = I
    lib.kvq_decode_attn_lost_wait_test.argtypes = [CP, P, I, I, I, P, I, P, I, ctypes.c_float, P, P,
                                                   Z, ctypes.c_uint32, ctypes.c_uint32, P]
    lib.kvq_compact_f16.restype = I
    lib.kvq_compact_f16.argtypes = [CP, P, I, P, P, P]
    lib.kvq_chunk_attn.restype = I
    lib.kvq_chunk_attn.argtypes = [P, P, I, I, I, P, I, I, ctypes.c_float, P, P]
    lib.kvq_chunk_attn_lost_wait_test.restype = I
    lib.kvq_chunk_attn_lost_wait_test.argtypes = [P, P, I, I, I, P, I, I, ctypes.c_float, P,
                                                  ctypes.c_uint32, ctypes.c_uint32, P]
    lib.kvq_gather_cells.restype = I
    lib.kvq_gather_cells.argtypes = [CP, P, I, P, P, P, P, P]
    lib.kvq_scatter_cells.restype = I
    lib.kvq_scatter_cells.argtypes = [CP, P, I, P, P, P, P, P]
    lib.kvq_stream_plan.restype = I
    lib.kvq_stream_plan.argtypes = [I, I, P, P, P, P, P, I, I, P, I, P, P, P, P, P]
    lib.kvq_stream_fetch.restype = I
    lib.kvq_stream_fetch.argtypes = [CP, CP, P, P, I, P]
    lib.kvq_decode_attn_static.restype = I
    lib.kvq_decode_attn_static.argtypes = [CP, P, I, I, I, P, I, P, I, ctypes.c_float, P, P]
    lib.kvq_status_string.restype = ctypes.c_char_p
    lib.kvq_status_string.argtypes = [I]
    if path is None:
        _lib = lib
    return lib


def _ptr(x):
    """Device (or host) address of a tensor / int / None."""
    if x is None:
        return None
    data_ptr = getattr(x, "data_ptr", None)   # torch tensors: the common case first
    if data_ptr is not None:
        return data_ptr()
    if isinstance(x, int):
        return x
    if hasattr(x, "ctypes") and hasattr(x, "dtype"):   # numpy (host) array
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


_current_stream = None   # () -> cudaStream_t of torch's current stream, set on first use


def _stream(stream):
    """cudaStream_t of a torch stream, an int handle, or (None) torch's
    current stream on the current device (read without building a Stream
    object, which costs a few microseconds a call)."""
    if stream is None:
        global _current_stream
        if _current_stream is None:
            import torch
            raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
            device = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device
            if raw is not None:
                _current_stream = lambda: raw(device())
            else:
                _current_stream = lambda: torch.cuda.current_stream().cuda_stream
        return _current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_cache(fmt: int, n_kv_heads: int, head_dim: int, block_size: int, n_blocks: int,
               k_data, v_data, k_scales=None, v_scales=None) -> kvq_cache:
    """Fill a kvq_cache from tensors (or raw device addresses)."""
    return kvq_cache(fmt, n_kv_heads, head_dim, block_size, n_blocks, 0,
                     _ptr(k_data), _ptr(v_data), _ptr(k_scales), _ptr(v_scales))


def kvq_block_bytes(fmt: int, n_kv_heads: int, head_dim: int, block_size: int) -> int:
    return int(load_library().kvq_block_bytes(fmt, n_kv_heads, head_dim, block_size))


def kvq_append(cache: kvq_cache, k, v, n_tok: int, tok_seq, tok_pos, block_table,
               n_seq: int, max_blocks_per_seq: int, stream=None) -> int:
    return load_library().kvq_append(ctypes.byref(cache), _ptr(k), _ptr(v), n_tok,
                                     _ptr(tok_seq), _ptr(tok_pos), _ptr(block_table),
                                     n_seq, max_blocks_per_seq, _stream(stream))


def kvq_decode_workspace_bytes(cache: kvq_cache, n_seq: int, W: int, n_q: int,
                               max_ctx: int) -> int:
    return int(load_library().kvq_decode_workspace_bytes(ctypes.byref(cache), n_seq, W, n_q,
                                                         max_ctx))


def kvq_decode_attn(cache: kvq_cache, q, n_seq: int, W: int, n_q: int, ctx_lens, max_ctx: int,
                    block_table, max_blocks_per_seq: int, sm_scale: float, out, workspace,
                    workspace_bytes: int, stream=None) -> int:
    return load_library().kvq_decode_attn(ctypes.byref(cache), _ptr(q), n_seq, W, n_q,
                                          _ptr(ctx_lens), max_ctx, _ptr(block_table),
                                          max_blocks_per_seq, float(sm_scale), _ptr(out),
                                          _ptr(workspace), int(workspace_bytes),
                                          _stream(stream))


def kvq_compact_f16(cache: kvq_cache, block_table_row, n_cells: int, out_k, out_v,
                    stream=None) -> int:
    return load_library().kvq_compact_f16(ctypes.byref(cache), _ptr(block_table_row), n_cells,
                                          _ptr(out_k), _ptr(out_v), _stream(stream))


def kvq_chunk_attn(k16, v16, n_kv_heads: int, P: int, head_dim: int, q, T: int, n_q: int,
                   sm_scale: float, out, stream=None) -> int:
    return load_library().kvq_chunk_attn(_ptr(k16), _ptr(v16), n_kv_heads, P, head_dim, _ptr(q),
                                         T, n_q, float(sm_scale), _ptr(out), _stream(stream))


def kvq_chunk_attn_lost_wait_test(k16, v16, n_kv_heads: int, P: int, head_dim: int, q, T: int,
                                  n_q: int, sm_scale: float, out, wait_limit: int,
                                  extra_tx_bytes: int, stream=None) -> int:
    return load_library().kvq_chunk_attn_lost_wait_test(
        _ptr(k16), _ptr(v16), n_kv_heads, P, head_dim, _ptr(q), T, n_q, float(sm_scale), _ptr(out),
        wait_limit, extra_tx_bytes, _stream(stream))


def kvq_gather_cells(cache: kvq_cache, block_table_row, n_cells: int, codes_k, codes_v,
                     scales_k=None, scales_v=None, stream=None) -> int:
    return load_library().kvq_gather_cells(ctypes.byref(cache), _ptr(block_table_row), n_cells,
                                           _ptr(codes_k), _ptr(codes_v), _ptr(scales_k),
                                           _ptr(scales_v), _stream(stream))


def kvq_scatter_cells(cache: kvq_cache, block_table_row, n_cells: int, codes_k, codes_v,
                      scales_k=None, scales_v=None, stream=None) -> int:
    return load_library().kvq_scatter_cells(ctypes.byref(cache), _ptr(block_table_row), n_cells,
                                            _ptr(codes_k), _ptr(codes_v), _ptr(scales_k),
                                            _ptr(scales_v), _stream(stream))


def kvq_decode_attn_static(cache: kvq_cache, q, n_seq: int, W: int, n_q: int, ctx_lens,
                           max_ctx: int, block_table, max_blocks_per_seq: int,
                           sm_scale: float, out, stream=None) -> int:
    """kvq_decode_attn with the library's own device scratch, for callers that
    cannot allocate (graph capture, framework-owned memory, fixed budgets)."""
    return load_library().kvq_decode_attn_static(ctypes.byref(cache), _ptr(q), n_seq, W, n_q,
                                                 _ptr(ctx_lens), max_ctx, _ptr(block_table),
                                                 max_blocks_per_seq, float(sm_scale), _ptr(out),
                                                 _stream(stream))


def kvq_stream_plan(n_host_blocks: int, n_slots: int, slot_of_block, block_of_slot, last_use,
                    clock, block_table, n_seq: int, max_blocks_per_seq: int, ctx_lens,
                    block_size: int, slot_table, fetch_src, fetch_dst, n_fetch, n_hits=None) -> int:
    """Host-only residency plan; every array argument is host memory (numpy
    arrays or CPU tensors); n_fetch / n_hits are 1-element int32 arrays."""
    return load_library().kvq_stream_plan(
        n_host_blocks, n_slots, _ptr(slot_of_block), _ptr(block_of_slot), _ptr(last_use),
        _ptr(clock), _ptr(block_table), n_seq, max_blocks_per_seq, _ptr(ctx_lens), block_size,
        _ptr(slot_table), _ptr(fetch_src), _ptr(fetch_dst), _ptr(n_fetch), _ptr(n_hits))


def kvq_stream_fetch(host_copy: kvq_cache, window: kvq_cache, fetch_src, fetch_dst,
                     n_fetch: int, stream=None) -> int:
    return load_library().kvq_stream_fetch(ctypes.byref(host_copy), ctypes.byref(window),
                                           _ptr(fetch_src), _ptr(fetch_dst), n_fetch,
                                           _stream(stream))


def kvq_decode_attn_lost_wait_test(cache: kvq_cache, q, n_seq: int, W: int, n_q: int, ctx_lens,
                                   max_ctx: int, block_table, max_blocks_per_seq: int,
                                   sm_scale: float, out, workspace, workspace_bytes: int,
                                   wait_limit: int, extra_tx_bytes: int, stream=None) -> int:
    return load_library().kvq_decode_attn_lost_wait_test(
        ctypes.byref(cache), _ptr(q), n_seq, W, n_q, _ptr(ctx_lens), max_ctx, _ptr(block_table),
        max_blocks_per_seq, float(sm_scale), _ptr(out), _ptr(workspace), workspace_bytes,
        wait_limit, extra_tx_bytes, _stream(stream))


def kvq_status_string(status: int) -> str:
    return load_library().kvq_status_string(int(status)).decode()


def check(status: int, where: str = "kvq") -> None:
    """Raise KvqError unless status is KVQ_OK."""
    if status != KVQ_OK:
        raise KvqError(status, where)

"""Save a sequence's cache to a file and restore it into a pool.

The file follows the shape of "Path F format v3: persist per-head INT8 KV
scales for INT8 + persistent KV interop" ("Scope"): a 128-byte header, the
saved cells' tokens, the K/V body, then -- new in version 3 -- the scales
body.  Its rules, from the same page ("Why", "Scope"): int8 codes are never
written or read without their scales, so an int8 pool refuses a version-2
file (which has no scales body); FP16 files need none.  The scales here are
this library's, one fp16 per 64 head dims per (cell, KV head), not the
per-head fp32 ones that page describes.

Layout (little-endian):
  header 128 B   magic b"KVQCELLS", version u32, format u32, n_kv u32,
                 head_dim u32, n_cells u32, group u32 (64), tokens_bytes u64,
                 body_bytes u64, scales_bytes u64, zeros to 128 B
  tokens         int32 [n_cells]
  body           codes_k then codes_v, each [n_cells][n_kv][head_dim]
                 (fp16 bits or int8; K8V4's codes_v [n_cells][n_kv][head_dim/2]
                 nibble bytes)
  scales         scales_k then scales_v, each [n_cells][n_kv][head_dim/64]
                 fp16 bits (int8 and K8V4; K8V4's scales_v per 32 dims)

The device side is kvq_gather_cells / kvq_scatter_cells (token-major runs,
bits unchanged); this module only moves their buffers to and from a file.
"""
from __future__ import annotations

import struct

import numpy as np

from . import (KVQ_F16, KVQ_GROUP, KVQ_K8V4, KVQ_Q4_BLOCK, KVQ_Q8, check, kvq_gather_cells,
               kvq_scatter_cells)

MAGIC = b"KVQCELLS"
VERSION = 3
HEADER_BYTES = 128
_HEAD = struct.Struct("<8sIIIIIIQQQ")


class CacheFileError(ValueError):
    """A cache file that cannot be restored into the given pool."""


def _layout(fmt: int, head_dim: int):
    """(K dtype, K elements per row, V dtype, V elements per row, K scales
    per row, V scales per row) of the runs of a format."""
    if fmt == KVQ_F16:
        return np.uint16, head_dim, np.uint16, head_dim, 0, 0
    if fmt == KVQ_Q8:
        return np.int8, head_dim, np.int8, head_dim, head_dim // KVQ_GROUP, head_dim // KVQ_GROUP
    if fmt == KVQ_K8V4:
        return (np.int8, head_dim, np.uint8, head_dim // 2, head_dim // KVQ_GROUP,
                head_dim // KVQ_Q4_BLOCK)
    raise CacheFileError(f"unknown cache format {fmt}")


def write_cells(path, fmt: int, n_kv: int, head_dim: int, tokens, codes_k, codes_v,
                scales_k=None, scales_v=None) -> None:
    """Write token-major runs (as kvq_gather_cells produces them) to `path`."""
    kdt, kn, vdt, vn, kng, vng = _layout(fmt, head_dim)
    codes_k = np.ascontiguousarray(codes_k).view(kdt)
    codes_v = np.ascontiguousarray(codes_v).view(vdt)
    n_cells = codes_k.shape[0]
    if codes_k.shape != (n_cells, n_kv, kn) or codes_v.shape != (n_cells, n_kv, vn):
        raise CacheFileError("codes do not have the format's shape [n_cells][n_kv][row]")
    if kng:
        if scales_k is None or scales_v is None:
            raise CacheFileError("int8 codes are never saved without their scales")
        scales_k = np.ascontiguousarray(scales_k).view(np.uint16)
        scales_v = np.ascontiguousarray(scales_v).view(np.uint16)
        if scales_k.shape != (n_cells, n_kv, kng) or scales_v.shape != (n_cells, n_kv, vng):
            raise CacheFileError("scales do not have the format's shape [n_cells][n_kv][groups]")
    tokens = np.zeros(n_cells, np.int32) if tokens is None else np.ascontiguousarray(tokens, np.int32)
    if tokens.shape != (n_cells,):
        raise CacheFileError("one token per saved cell")
    body = codes_k.nbytes + codes_v.nbytes
    sbytes = scales_k.nbytes + scales_v.nbytes if kng else 0
    head = _HEAD.pack(MAGIC, VERSION, fmt, n_kv, head_dim, n_cells, KVQ_GROUP, tokens.nbytes,
                      body, sbytes)
    with open(path, "wb") as f:
        f.write(head + b"\0" * (HEADER_BYTES - len(head)))
        f.write(tokens.tobytes())
        f.write(codes_k.tobytes())
        f.write(codes_v.tobytes())
        if kng:
            f.write(scales_k.tobytes())
            f.write(scales_v.tobytes())


def read_cells(path, fmt: int, n_kv: int, head_dim: int):
    """Read a file written by write_cells for a pool of the given format and
    geometry; returns (tokens, codes_k, codes_v, scales_k, scales_v).
    Raises CacheFileError when the file cannot be restored into such a pool."""
    with open(path, "rb") as f:
        raw = f.read()
    if len(raw) < HEADER_BYTES:
        raise CacheFileError("file shorter than its header")
    magic, version, ffmt, fkv, fhd, n_cells, group, tbytes, body, sbytes = _HEAD.unpack_from(raw)
    if magic != MAGIC:
        raise CacheFileError("not a cache file")
    if version not in (2, 3):
        raise CacheFileError(f"unsupported version {version}")
    if ffmt != fmt or fkv != n_kv or fhd != head_dim:
        raise CacheFileError("file format or geometry differs from the pool's")
    if group != KVQ_GROUP:
        raise CacheFileError(f"scale group of {group} dims, this library uses {KVQ_GROUP}")
    kdt, kn, vdt, vn, kng, vng = _layout(fmt, head_dim)
    if kng and (version < 3 or sbytes == 0):
        raise CacheFileError("int8 codes without their scales: refusing to restore")
    rows = n_cells * n_kv
    kbytes = rows * kn * np.dtype(kdt).itemsize
    want_body = kbytes + rows * vn * np.dtype(vdt).itemsize
    want_s = rows * (kng + vng) * 2
    if tbytes != 4 * n_cells or body != want_body or sbytes != want_s:
        raise CacheFileError("section sizes do not match the header")
    if len(raw) != HEADER_BYTES + tbytes + body + sbytes:
        raise CacheFileError("file length does not match the header")
    at = HEADER_BYTES
    tokens = np.frombuffer(raw, np.int32, n_cells, at)
    at += tbytes
    codes_k = np.frombuffer(raw, kdt, rows * kn, at).reshape(n_cells, n_kv, kn)
    codes_v = np.frombuffer(raw, vdt, rows * vn, at + kbytes).reshape(n_cells, n_kv, vn)
    at += body
    scales_k = scales_v = None
    if kng:
        scales_k = np.frombuffer(raw, np.uint16, rows * kng, at).reshape(n_cells, n_kv, kng)
        scales_v = np.frombuffer(raw, np.uint16, rows * vng, at + rows * kng * 2).reshape(
            n_cells, n_kv, vng)
    return tokens.copy(), codes_k.copy(), codes_v.copy(), \
        None if scales_k is None else scales_k.copy(), None if scales_v is None else scales_v.copy()


def save_sequence(path, pool, block_table_row, n_cells: int, tokens=None, stream=None) -> None:
    """Gather cells [0, n_cells) of one sequence of a PagedPool (device) and
    write them to `path`."""
    import torch

    from .pool import on_stream, row_layout

    dev = pool.k.device
    kdt, kn, vdt, vn, kng, vng = row_layout(pool.fmt, pool.head_dim)
    with on_stream(stream):
        ck = torch.empty((n_cells, pool.n_kv, kn), dtype=kdt, device=dev)
        cv = torch.empty((n_cells, pool.n_kv, vn), dtype=vdt, device=dev)
        sk = sv = None
        if kng:
            sk = torch.empty((n_cells, pool.n_kv, kng), dtype=torch.float16, device=dev)
            sv = torch.empty((n_cells, pool.n_kv, vng), dtype=torch.float16, device=dev)
        check(kvq_gather_cells(pool.cache, block_table_row, n_cells, ck, cv, sk, sv, stream),
              "kvq_gather_cells")
    torch.cuda.synchronize(dev)  # the gather may run on a stream of the caller's
    host = lambda t: None if t is None else t.cpu().numpy()
    bits = lambda a: None if a is None else (a.view(np.uint16) if a.dtype == np.float16 else a)
    write_cells(path, pool.fmt, pool.n_kv, pool.head_dim, tokens, bits(host(ck)), bits(host(cv)),
                bits(host(sk)), bits(host(sv)))


def load_sequence(path, pool, block_table_row, stream=None):
    """Restore a file written by save_sequence into a PagedPool under the
    given block-table row; returns (n_cells, tokens)."""
    import torch

    from .pool import on_stream

    tokens, ck, cv, sk, sv = read_cells(path, pool.fmt, pool.n_kv, pool.head_dim)
    dev = pool.k.device
    to_dev = lambda a, dt: None if a is None else torch.from_numpy(a.view(dt)).to(dev)
    cdt = np.float16 if pool.fmt == KVQ_F16 else np.int8
    n_cells = ck.shape[0]
    with on_stream(stream):   # the staging copies run on the scatter's stream, ahead of it
        dk, dv = to_dev(ck, cdt), to_dev(cv, cdt if pool.fmt != KVQ_K8V4 else np.uint8)
        dsk, dsv = to_dev(sk, np.float16), to_dev(sv, np.float16)
        check(kvq_scatter_cells(pool.cache, block_table_row, n_cells, dk, dv, dsk, dsv, stream),
              "kvq_scatter_cells")
    torch.cuda.synchronize(dev)  # the staging tensors live until the scatter has run
    return n_cells, tokens

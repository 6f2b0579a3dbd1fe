"""A paged K/V pool held in torch device tensors, driven through the C ABI.

PyTorch only provides the device memory and the stream here; every step of
append, decode attention and compaction runs in libkvq.so.  The methods are
argument marshalling over the entry points of the same names.
"""
from __future__ import annotations

import contextlib

import torch

from . import (KVQ_F16, KVQ_GROUP, KVQ_K8V4, KVQ_Q4_BLOCK, KVQ_Q8, check, kvq_append,
               kvq_compact_f16, kvq_decode_attn, kvq_decode_workspace_bytes, make_cache)


def on_stream(stream):
    """Context under which tensors allocated for a call belong to the stream
    the call runs on (torch's allocator then never hands their memory to
    other work before that stream reaches it).  None: torch's current
    stream, which allocations use already."""
    if stream is None:
        return contextlib.nullcontext()
    if isinstance(stream, int):
        stream = torch.cuda.ExternalStream(stream)
    return torch.cuda.stream(stream)


def row_layout(fmt: int, head_dim: int):
    """(K dtype, K elements per row, V dtype, V elements per row, K scales
    per row, V scales per row) of one pool row in the given format."""
    if fmt == KVQ_F16:
        return torch.float16, head_dim, torch.float16, head_dim, 0, 0
    if fmt == KVQ_Q8:
        return torch.int8, head_dim, torch.int8, head_dim, head_dim // KVQ_GROUP, head_dim // KVQ_GROUP
    if fmt == KVQ_K8V4:   # V: two 4-bit codes a byte, one scale per 32 rotated dims
        return (torch.int8, head_dim, torch.uint8, head_dim // 2, head_dim // KVQ_GROUP,
                head_dim // KVQ_Q4_BLOCK)
    raise ValueError(f"unknown cache format {fmt}")


class PagedPool:
    """One layer's pool: codes [n_blocks][n_kv][bs][hd] (+ fp16 scales for int8;
    K8V4: int8 K, V nibbles [..][hd/2], V scales [..][hd/32])."""

    def __init__(self, fmt: int, n_kv: int, head_dim: int, block_size: int, n_blocks: int,
                 device="cuda", fill: int = 0, pinned: bool = False):
        """pinned: hold the arrays in pinned host memory (a streaming host
        copy, which the kernels address directly) instead of on `device`."""
        self.fmt, self.n_kv, self.head_dim = fmt, n_kv, head_dim
        self.block_size, self.n_blocks = block_size, n_blocks
        kdt, kn, vdt, vn, kng, vng = row_layout(fmt, head_dim)
        lead = (n_blocks, n_kv, block_size)
        where = dict(device="cpu", pin_memory=True) if pinned else dict(device=device)

        def make(n, dt):
            t = torch.zeros(lead + (n,), dtype=dt, **where)
            if fill:
                t.fill_(fill)
            return t

        self.k = make(kn, kdt)
        self.v = make(vn, vdt)
        self.ks = make(kng, torch.float16) if kng else None
        self.vs = make(vng, torch.float16) if vng else None
        self.cache = make_cache(fmt, n_kv, head_dim, block_size, n_blocks,
                                self.k, self.v, self.ks, self.vs)

    def append(self, k, v, tok_seq, tok_pos, block_table, stream=None) -> None:
        n_tok = int(tok_seq.shape[0])
        check(kvq_append(self.cache, k, v, n_tok, tok_seq, tok_pos, block_table,
                         int(block_table.shape[0]), int(block_table.shape[1]), stream),
              "kvq_append")

    def workspace_bytes(self, n_seq: int, W: int, n_q: int, max_ctx: int) -> int:
        return kvq_decode_workspace_bytes(self.cache, n_seq, W, n_q, max_ctx)

    def decode(self, q, ctx_lens, max_ctx: int, block_table, sm_scale: float, out=None,
               workspace=None, stream=None):
        n_seq, W, n_q, hd = q.shape
        with on_stream(stream):
            if out is None:
                out = torch.empty_like(q)
            if workspace is None:   # needs no initial contents; a given one is checked by the call
                need = self.workspace_bytes(n_seq, W, n_q, max_ctx)
                workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
            check(kvq_decode_attn(self.cache, q, n_seq, W, n_q, ctx_lens, max_ctx, block_table,
                                  int(block_table.shape[1]), sm_scale, out, workspace,
                                  workspace.numel(), stream), "kvq_decode_attn")
        return out

    def compact(self, block_table_row, n_cells: int, out_k=None, out_v=None, stream=None):
        shape = (self.n_kv, n_cells, self.head_dim)
        with on_stream(stream):
            if out_k is None:
                out_k = torch.empty(shape, dtype=torch.float16, device=self.k.device)
            if out_v is None:
                out_v = torch.empty(shape, dtype=torch.float16, device=self.k.device)
            check(kvq_compact_f16(self.cache, block_table_row, n_cells, out_k, out_v, stream),
                  "kvq_compact_f16")
        return out_k, out_v

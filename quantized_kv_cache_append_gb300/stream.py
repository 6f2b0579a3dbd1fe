"""A streamed pool: the authoritative cache in pinned host memory and a
resident window of device blocks, driven through kvq_stream_plan /
kvq_stream_fetch (include/kvq.h).

#711 kv: --kv k8v4 streams with --kv-resident, "What" and "How": the host
copy holds every cell; the window holds N cells' worth of blocks; appends
write both; attention reads the window under the slot table.  This module
is argument marshalling: the plan runs in the library's host code, the
fetch and every append / attention in its kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import check, kvq_stream_fetch, kvq_stream_plan
from .pool import PagedPool, on_stream


class StreamedPool:
    """Host copy of n_host_blocks blocks (pinned) + a window of n_slots
    device blocks + the residency state (host arrays)."""

    def __init__(self, fmt: int, n_kv: int, head_dim: int, block_size: int, n_host_blocks: int,
                 n_slots: int, device="cuda"):
        self.block_size, self.n_host_blocks, self.n_slots = block_size, n_host_blocks, n_slots
        self.host = PagedPool(fmt, n_kv, head_dim, block_size, n_host_blocks, pinned=True)
        self.window = PagedPool(fmt, n_kv, head_dim, block_size, n_slots, device=device)
        self.slot_of_block = np.full(n_host_blocks, -1, np.int32)
        self.block_of_slot = np.full(n_slots, -1, np.int32)
        self.last_use = np.zeros(n_slots, np.int64)
        self.clock = np.zeros(1, np.int64)
        self._src = np.zeros(n_slots, np.int32)
        self._dst = np.zeros(n_slots, np.int32)
        self._n = np.zeros(2, np.int32)
        self.device = device
        # the host copy must be device-addressable before anything writes to it
        check(kvq_stream_fetch(self.host.cache, self.window.cache, None, None, 0), "kvq_stream_fetch")

    def append_host(self, k, v, tok_seq, tok_pos, block_table_dev, stream=None) -> None:
        """The authoritative write (host copy, host block ids)."""
        self.host.append(k, v, tok_seq, tok_pos, block_table_dev, stream)

    def plan(self, block_table: np.ndarray, ctx_lens: np.ndarray):
        """Host plan for one call; returns (slot_table host array, fetch
        pairs (src, dst) as host arrays, hits)."""
        bt = np.ascontiguousarray(block_table, np.int32)
        ctx = np.ascontiguousarray(ctx_lens, np.int32)
        slot_table = np.empty_like(bt)
        check(kvq_stream_plan(self.n_host_blocks, self.n_slots, self.slot_of_block,
                              self.block_of_slot, self.last_use, self.clock, bt, bt.shape[0],
                              bt.shape[1], ctx, self.block_size, slot_table, self._src, self._dst,
                              self._n[:1], self._n[1:]), "kvq_stream_plan")
        n = int(self._n[0])
        return slot_table, self._src[:n].copy(), self._dst[:n].copy(), int(self._n[1])

    def fetch(self, src: np.ndarray, dst: np.ndarray, stream=None) -> None:
        """Copy the planned blocks from the host copy into their slots."""
        if len(src) == 0:
            return
        with on_stream(stream):   # the id copies run on the fetch's own stream, ahead of it
            d_src = torch.from_numpy(np.ascontiguousarray(src, np.int32)).to(self.device)
            d_dst = torch.from_numpy(np.ascontiguousarray(dst, np.int32)).to(self.device)
            check(kvq_stream_fetch(self.host.cache, self.window.cache, d_src, d_dst, len(src),
                                   stream), "kvq_stream_fetch")
        self._keep = (d_src, d_dst)   # alive until the next fetch is queued behind this one

"""Seeded synthetic inputs for the five K/V-cache workloads.

This module only draws random numbers and lays out block tables; it holds
none of the method's arithmetic (no rounding, quantization or attention), so
that the CUDA path and the CPU oracle can both be fed from it without
sharing any of their computation.

Workloads (fp32 K/V/Q, N(0,1) unless stated):
  tiny          1 sequence, 4 query / 1 KV heads, head_dim 128, 1024 cells,
                1 decode token; FP16 and int8 caches.
  gqa32k        1 sequence, 32 / 8 heads, head_dim 128, 32768 cells prefilled,
                then 64 steps of (append 1 cell, decode 1 token).  K has 4
                outlier channels per KV head, scaled x20 for every cell.
  ragged        16 sequences, lengths uniform in [1024, 16384], 32 / 8 heads,
                head_dim 128, int8 cache, 1 decode token per sequence.
  long256k      1 sequence, 16 / 2 heads, head_dim 256 (4 scale groups),
                262144 cells; 1% of (cell, KV head) rows have K and V x10.
  chunk_verify  126976 cells prefilled, a 4096-cell chunk appended (int8) to
                reach 131072, FP16 compaction of all 131072 cells, then a
                4-token causal verify window; 32 / 8 heads, head_dim 128.

Every workload uses block size 256 and one seeded shuffled permutation of the
physical blocks (the block table maps logical blocks to shuffled physical
ones).  Seed = 1000 + the workload's number (1..5).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np
import torch

BLOCK_SIZE = 256

WORKLOADS = ("tiny", "gqa32k", "ragged", "long256k", "chunk_verify")
WORKLOAD_NUMBER = {name: i + 1 for i, name in enumerate(WORKLOADS)}


@dataclasses.dataclass
class Workload:
    name: str
    n_kv: int
    head_dim: int
    n_q: int
    W: int
    block_size: int
    n_seq: int
    formats: tuple
    # cells present before the timed/checked step, per sequence
    ctx_lens: np.ndarray                 # int32 [n_seq] (after the prefill)
    block_table: np.ndarray              # int32 [n_seq][max_blocks]
    n_blocks: int
    # prefill: the cells written before decoding
    k: np.ndarray                        # float32 [n_tok][n_kv][hd]
    v: np.ndarray
    tok_seq: np.ndarray                  # int32 [n_tok]
    tok_pos: np.ndarray                  # int32 [n_tok]
    q: np.ndarray                        # float32 [n_seq][W][n_q][hd]
    sm_scale: float
    # optional: cells appended in a second call (chunk_verify) ...
    chunk: Optional[Dict[str, np.ndarray]] = None
    # ... or per-step appends + queries (gqa32k): list of dicts
    steps: Optional[List[Dict[str, np.ndarray]]] = None
    # structure of the draw (outlier channels / rows), for checks and docs
    extra: Optional[Dict[str, np.ndarray]] = None

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _randn(g: torch.Generator, *shape) -> np.ndarray:
    return torch.randn(*shape, generator=g, dtype=torch.float32).numpy()


def _block_table(g: torch.Generator, capacities, block_size: int):
    """Logical blocks of every sequence mapped to one shuffled physical order."""
    nb_per_seq = [max(1, math.ceil(c / block_size)) for c in capacities]
    n_blocks = int(sum(nb_per_seq))
    perm = torch.randperm(n_blocks, generator=g).numpy().astype(np.int32)
    max_blocks = max(nb_per_seq)
    table = np.full((len(capacities), max_blocks), -1, dtype=np.int32)
    at = 0
    for b, nb in enumerate(nb_per_seq):
        table[b, :nb] = perm[at:at + nb]
        at += nb
    return table, n_blocks


def _prefill_positions(lens):
    seq = np.concatenate([np.full(L, b, dtype=np.int32) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    return seq, pos


def sm_scale_for(head_dim: int) -> float:
    return float(np.float32(1.0) / np.sqrt(np.float32(head_dim)))


def make(name: str, *, scale_cells: float = 1.0) -> Workload:
    """Build a workload.  scale_cells < 1 shrinks every context length (for
    quick tests); the shapes, distributions and structure stay the same."""
    if name not in WORKLOAD_NUMBER:
        raise KeyError(name)
    seed = 1000 + WORKLOAD_NUMBER[name]
    g = _gen(seed)
    bs = BLOCK_SIZE

    def cells(n):
        return max(1, int(round(n * scale_cells)))

    if name == "tiny":
        n_kv, hd, n_q, W, L = 1, 128, 4, 1, cells(1024)
        lens = [L]
        k = _randn(g, L, n_kv, hd)
        v = _randn(g, L, n_kv, hd)
        q = _randn(g, 1, W, n_q, hd)
        table, nb = _block_table(g, lens, bs)
        seq, pos = _prefill_positions(lens)
        return Workload(name, n_kv, hd, n_q, W, bs, 1, ("f16", "q8"),
                        np.array(lens, np.int32), table, nb, k, v, seq, pos, q,
                        sm_scale_for(hd))

    if name == "gqa32k":
        n_kv, hd, n_q, W, L, n_steps = 8, 128, 32, 1, cells(32768), 64
        k = _randn(g, L, n_kv, hd)
        v = _randn(g, L, n_kv, hd)
        q = _randn(g, 1, W, n_q, hd)
        # 4 outlier channels per KV head, K scaled x20 in every cell
        chans = np.stack([torch.randperm(hd, generator=g)[:4].numpy() for _ in range(n_kv)])
        step_k = _randn(g, n_steps, 1, n_kv, hd)
        step_v = _randn(g, n_steps, 1, n_kv, hd)
        step_q = _randn(g, n_steps, 1, W, n_q, hd)
        for h in range(n_kv):
            k[:, h, chans[h]] *= 20.0
            step_k[:, :, h, chans[h]] *= 20.0
        table, nb = _block_table(g, [L + n_steps], bs)
        seq, pos = _prefill_positions([L])
        steps = []
        for i in range(n_steps):
            steps.append(dict(k=step_k[i], v=step_v[i], q=step_q[i],
                              tok_seq=np.zeros(1, np.int32),
                              tok_pos=np.array([L + i], np.int32),
                              ctx_lens=np.array([L + i + 1], np.int32)))
        return Workload(name, n_kv, hd, n_q, W, bs, 1, ("f16", "q8"),
                        np.array([L], np.int32), table, nb, k, v, seq, pos, q,
                        sm_scale_for(hd), steps=steps, extra=dict(outlier_channels=chans))

    if name == "ragged":
        n_kv, hd, n_q, W, n_seq = 8, 128, 32, 1, 16
        lo, hi = cells(1024), cells(16384)
        lens = torch.randint(lo, hi + 1, (n_seq,), generator=g).numpy().astype(np.int32)
        n_tok = int(lens.sum())
        k = _randn(g, n_tok, n_kv, hd)
        v = _randn(g, n_tok, n_kv, hd)
        q = _randn(g, n_seq, W, n_q, hd)
        table, nb = _block_table(g, list(lens), bs)
        seq, pos = _prefill_positions(list(lens))
        return Workload(name, n_kv, hd, n_q, W, bs, n_seq, ("q8",),
                        lens, table, nb, k, v, seq, pos, q, sm_scale_for(hd))

    if name == "long256k":
        n_kv, hd, n_q, W, L = 2, 256, 16, 1, cells(262144)
        k = _randn(g, L, n_kv, hd)
        v = _randn(g, L, n_kv, hd)
        q = _randn(g, 1, W, n_q, hd)
        # 1% of (cell, KV head) rows: K and V scaled x10
        mask = (torch.rand(L, n_kv, generator=g) < 0.01).numpy()
        k[mask] *= 10.0
        v[mask] *= 10.0
        table, nb = _block_table(g, [L], bs)
        seq, pos = _prefill_positions([L])
        return Workload(name, n_kv, hd, n_q, W, bs, 1, ("f16", "q8"),
                        np.array([L], np.int32), table, nb, k, v, seq, pos, q,
                        sm_scale_for(hd), extra=dict(outlier_rows=mask))

    # chunk_verify
    n_kv, hd, n_q, W = 8, 128, 32, 4
    chunk_len = cells(4096)
    prefill = cells(131072) - chunk_len
    L = prefill + chunk_len
    k = _randn(g, prefill, n_kv, hd)
    v = _randn(g, prefill, n_kv, hd)
    ck = _randn(g, chunk_len, n_kv, hd)
    cv = _randn(g, chunk_len, n_kv, hd)
    q = _randn(g, 1, W, n_q, hd)
    table, nb = _block_table(g, [L], bs)
    seq, pos = _prefill_positions([prefill])
    chunk = dict(k=ck, v=cv, tok_seq=np.zeros(chunk_len, np.int32),
                 tok_pos=np.arange(prefill, L, dtype=np.int32),
                 ctx_lens=np.array([L], np.int32))
    return Workload(name, n_kv, hd, n_q, W, bs, 1, ("q8",),
                    np.array([prefill], np.int32), table, nb, k, v, seq, pos, q,
                    sm_scale_for(hd), chunk=chunk)

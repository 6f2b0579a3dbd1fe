"""The seeded synthetic inputs (workloads.py) follow the recipe the parity
tests and the bench rely on: the same draw for the same workload, the
stated shapes and sizes, block tables that map every logical block to a
distinct physical one, and the stated structure (outlier channels of
gqa32k, outlier rows of long256k, ragged lengths, the chunk of
chunk_verify).  CPU only."""
import numpy as np
import pytest

import workloads

SMALL = 1.0 / 32   # shrinks the long contexts; shapes and structure stay


def _table_ok(wl):
    t = wl.block_table
    used = [t[b, : -(-int(n) // wl.block_size)] for b, n in enumerate(wl.ctx_lens)]
    ids = np.concatenate(used)
    assert ids.min() >= 0 and ids.max() < wl.n_blocks
    assert len(np.unique(ids)) == len(ids)            # no physical block shared
    assert not np.array_equal(ids, np.sort(ids))      # shuffled, not the identity


@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_same_seed_same_draw(name):
    a, b = workloads.make(name, scale_cells=SMALL), workloads.make(name, scale_cells=SMALL)
    for x, y in ((a.k, b.k), (a.v, b.v), (a.q, b.q), (a.block_table, b.block_table)):
        assert np.array_equal(x, y)


def test_tiny_and_gqa32k_shapes():
    t = workloads.make("tiny")
    assert (t.n_kv, t.head_dim, t.n_q, t.W, int(t.ctx_lens[0])) == (1, 128, 4, 1, 1024)
    assert t.k.shape == (1024, 1, 128) and t.k.dtype == np.float32
    g = workloads.make("gqa32k", scale_cells=SMALL)
    assert (g.n_kv, g.head_dim, g.n_q, g.W, g.block_size) == (8, 128, 32, 1, 256)
    assert len(g.steps) == 64
    L = int(g.ctx_lens[0])
    for i, st in enumerate(g.steps):
        assert int(st["tok_pos"][0]) == L + i and int(st["ctx_lens"][0]) == L + i + 1
    _table_ok(g)
    assert abs(g.sm_scale - 1.0 / np.sqrt(128)) < 1e-7


def test_gqa32k_outlier_channels_are_scaled_by_20():
    g = workloads.make("gqa32k", scale_cells=SMALL)
    chans = g.extra["outlier_channels"]
    assert chans.shape == (8, 4)
    for h in range(8):
        sd = g.k[:, h, :].std(axis=0)
        out = np.zeros(128, bool)
        out[chans[h]] = True
        assert np.all(sd[out] > 15.0) and np.all(sd[~out] < 1.3)
    assert g.v.std() < 1.1                              # V untouched


def test_ragged_lengths_and_tables():
    r = workloads.make("ragged")
    assert r.n_seq == 16 and r.formats == ("q8",)
    assert r.ctx_lens.min() >= 1024 and r.ctx_lens.max() <= 16384
    assert r.k.shape[0] == int(r.ctx_lens.sum())
    _table_ok(r)


def test_long256k_outlier_rows():
    w = workloads.make("long256k", scale_cells=SMALL)
    assert (w.n_kv, w.head_dim, w.n_q) == (2, 256, 16)
    mask = w.extra["outlier_rows"]
    assert 0.005 < mask.mean() < 0.015                  # about 1 % of rows
    assert w.k[mask].std() > 8.0 and w.k[~mask].std() < 1.1
    assert w.v[mask].std() > 8.0


def test_chunk_verify_layout():
    c = workloads.make("chunk_verify", scale_cells=SMALL)
    chunk = c.chunk
    pre, L = int(c.ctx_lens[0]), int(chunk["ctx_lens"][0])   # before / after the chunk
    assert c.W == 4 and c.k.shape[0] == pre and pre + chunk["k"].shape[0] == L
    assert np.array_equal(chunk["tok_pos"], np.arange(pre, L, dtype=np.int32))
    full = workloads.make("chunk_verify")
    assert int(full.chunk["ctx_lens"][0]) == 131072 and full.chunk["k"].shape[0] == 4096
    assert int(full.ctx_lens[0]) == 126976

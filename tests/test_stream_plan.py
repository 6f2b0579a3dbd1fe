"""The residency plan of the streamed pool, on the CPU (host code only).

#711 kv: --kv k8v4 streams with --kv-resident, "What" and "Measured": a
window of N cells' worth of device blocks serves the blocks each call reads
(hits), and the others are fetched from the host copy (misses).  The
library's kvq_stream_plan is checked against a model of the policy written
here from its definition in include/kvq.h (hits keep their slots; misses
take free slots in index order, then the least recently used slots that
the call does not read, ties by index), step by step over random batches,
and against the policy's invariants.
"""
import numpy as np
import pytest

import quantized_kv_cache_append_gb300 as kvq


class Model:
    def __init__(self, n_blocks, n_slots):
        self.nb, self.ns = n_blocks, n_slots
        self.slot_of = [-1] * n_blocks
        self.block_of = [-1] * n_slots
        self.last = [0] * n_slots
        self.clock = 0

    def plan(self, table, ctx, bs):
        need, seen = [], set()
        for b, L in enumerate(ctx):
            for j in range(-(-int(L) // bs)):
                blk = int(table[b][j])
                if 0 <= blk < self.nb and blk not in seen:
                    seen.add(blk)
                    need.append(blk)
        if len(need) > self.ns:
            return None
        self.clock += 1
        hits = [x for x in need if self.slot_of[x] >= 0 and self.block_of[self.slot_of[x]] == x]
        for x in hits:
            self.last[self.slot_of[x]] = self.clock
        misses = [x for x in need if x not in set(hits)]
        free = [s for s in range(self.ns) if self.block_of[s] < 0]
        old = sorted((s for s in range(self.ns) if self.block_of[s] >= 0 and self.last[s] != self.clock),
                     key=lambda s: (self.last[s], s))
        fetch = []
        for x, s in zip(misses, free + old):
            if self.block_of[s] >= 0:
                self.slot_of[self.block_of[s]] = -1
            self.block_of[s], self.slot_of[x], self.last[s] = x, s, self.clock
            fetch.append((x, s))
        st = [[self.slot_of[int(x)] if 0 <= int(x) < self.nb else -1 for x in row] for row in table]
        return np.array(st, np.int32), fetch, len(hits)


class Lib:
    def __init__(self, n_blocks, n_slots):
        self.nb, self.ns = n_blocks, n_slots
        self.slot_of = np.full(n_blocks, -1, np.int32)
        self.block_of = np.full(n_slots, -1, np.int32)
        self.last = np.zeros(n_slots, np.int64)
        self.clock = np.zeros(1, np.int64)

    def plan(self, table, ctx, bs):
        table = np.ascontiguousarray(table, np.int32)
        ctx = np.ascontiguousarray(ctx, np.int32)
        st = np.empty_like(table)
        src = np.zeros(self.ns, np.int32)
        dst = np.zeros(self.ns, np.int32)
        n = np.zeros(1, np.int32)
        hits = np.zeros(1, np.int32)
        rc = kvq.kvq_stream_plan(self.nb, self.ns, self.slot_of, self.block_of, self.last,
                                 self.clock, table, table.shape[0], table.shape[1], ctx, bs, st,
                                 src, dst, n, hits)
        if rc == kvq.KVQ_ERR_UNSUPPORTED:
            return None
        assert rc == kvq.KVQ_OK, kvq.kvq_status_string(rc)
        return st, list(zip(src[: n[0]].tolist(), dst[: n[0]].tolist())), int(hits[0])


def _tables(rng, n_seq, max_blocks, n_blocks):
    perm = rng.permutation(n_blocks).astype(np.int32)
    return perm[: n_seq * max_blocks].reshape(n_seq, max_blocks)


@pytest.mark.parametrize("n_slots,seed", [(6, 1), (16, 2), (40, 3), (64, 4)])
def test_plan_matches_the_policy_model(n_slots, seed):
    rng = np.random.default_rng(seed)
    bs, n_seq, max_blocks = 16, 12, 8
    n_blocks = n_seq * max_blocks + 5
    table = _tables(rng, n_seq, max_blocks, n_blocks)
    lens = rng.integers(1, max_blocks * bs, n_seq)
    model, lib = Model(n_blocks, n_slots), Lib(n_blocks, n_slots)
    refused = fetched = hit = 0
    for step in range(300):
        batch = rng.choice(n_seq, size=int(rng.integers(1, 4)), replace=False)
        lens[batch] = np.minimum(lens[batch] + rng.integers(0, 3, len(batch)), max_blocks * bs)
        t, ctx = table[batch], lens[batch]
        a, b = model.plan(t, ctx, bs), lib.plan(t, ctx, bs)
        if a is None:
            assert b is None
            refused += 1
            continue
        np.testing.assert_array_equal(b[0], a[0])
        assert b[1] == a[1] and b[2] == a[2]
        fetched += len(b[1])
        hit += b[2]
        # the state arrays agree too
        assert lib.slot_of.tolist() == model.slot_of and lib.block_of.tolist() == model.block_of
    assert fetched > 0 and hit > 0
    if n_slots == 6:
        assert refused > 0


def test_invariants_and_refusal_leaves_state_unchanged():
    rng = np.random.default_rng(7)
    bs, n_blocks, n_slots = 32, 50, 10
    lib = Lib(n_blocks, n_slots)
    for _ in range(200):
        n_seq = int(rng.integers(1, 4))
        table = rng.integers(-2, n_blocks + 2, (n_seq, 6)).astype(np.int32)   # some ids out of range
        ctx = rng.integers(0, 6 * bs + 1, n_seq).astype(np.int32)
        before = (lib.slot_of.copy(), lib.block_of.copy(), lib.last.copy(), lib.clock.copy())
        r = lib.plan(table, ctx, bs)
        need = {int(table[b, j]) for b in range(n_seq) for j in range(-(-int(ctx[b]) // bs))
                if 0 <= table[b, j] < n_blocks}
        if r is None:
            assert len(need) > n_slots
            for x, y in zip(before, (lib.slot_of, lib.block_of, lib.last, lib.clock)):
                np.testing.assert_array_equal(x, y)
            continue
        st, fetch, hits = r
        assert hits + len(fetch) == len(need)
        assert len({s for _, s in fetch}) == len(fetch)                      # distinct slots
        for blk in need:                                                      # all resident
            s = lib.slot_of[blk]
            assert 0 <= s < n_slots and lib.block_of[s] == blk
        for b in range(n_seq):
            for j in range(-(-int(ctx[b]) // bs)):
                blk = int(table[b, j])
                assert st[b, j] == (lib.slot_of[blk] if 0 <= blk < n_blocks else -1)
        occupied = lib.block_of[lib.block_of >= 0]
        assert len(set(occupied.tolist())) == len(occupied)                  # one slot per block


def test_a_window_as_large_as_the_working_set_stops_missing():
    bs, n_blocks = 16, 40
    table = np.arange(40, dtype=np.int32).reshape(4, 10)
    ctx = np.full(4, 10 * bs, np.int32)
    lib = Lib(n_blocks, 40)
    first = lib.plan(table, ctx, bs)
    assert len(first[1]) == 40 and first[2] == 0
    again = lib.plan(table, ctx, bs)
    assert len(again[1]) == 0 and again[2] == 40


def test_plan_argument_checks():
    z = np.zeros(4, np.int32)
    args = lambda **kw: dict(dict(nb=8, ns=4, bs=16, n_seq=1, mb=1), **kw)
    def call(**kw):
        a = args(**kw)
        st = np.zeros(max(a["n_seq"], 1) * a["mb"], np.int32)
        return kvq.kvq_stream_plan(a["nb"], a["ns"], np.full(8, -1, np.int32),
                                   np.full(4, -1, np.int32), np.zeros(4, np.int64),
                                   np.zeros(1, np.int64), np.zeros(4, np.int32), a["n_seq"], a["mb"],
                                   np.full(4, a.get("ctx", 16), np.int32), a["bs"], st, z.copy(),
                                   z.copy(), np.zeros(1, np.int32), None)
    assert call() == kvq.KVQ_OK
    assert call(nb=0) == kvq.KVQ_ERR_ARG
    assert call(ns=0) == kvq.KVQ_ERR_ARG
    assert call(bs=0) == kvq.KVQ_ERR_ARG
    assert call(ctx=17) == kvq.KVQ_ERR_ARG          # beyond the row's blocks
    assert call(n_seq=0) == kvq.KVQ_OK               # nothing to read

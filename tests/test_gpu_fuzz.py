"""GPU parity over seeded random shapes: append, decode attention and
compaction of every format against the oracle.

Each case draws a head dim, block size, KV head count, GQA group, verify
window, a batch of ragged lengths (some empty, some one block plus one
cell), a shuffled block table with spare blocks, and inputs with scaled
rows; the appends arrive in several calls of random sizes (decode-step and
bulk kernel shapes alike).  Bars as everywhere: cache bytes and compaction
bit-exact, attention within max-abs 2e-3 and relative L2 1e-3.
"""
import numpy as np
import pytest
import torch

import workloads
import quantized_kv_cache_append_gb300 as kvq
from tests.gpu_pairs import Pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("the GPU suite needs a CUDA device")
    kvq.build()
    kvq.load_library()


def _case(seed):
    rng = np.random.default_rng(seed)
    fmt = ["f16", "q8", "k8v4"][seed % 3]
    hd = int(rng.choice([64, 128, 256]))
    bs = int(rng.choice([16, 32, 64, 256, 1024]))
    n_kv = int(rng.choice([1, 2, 3, 4, 8]))
    max_rows = 32   # rows beyond one CTA's tile (16 at head_dim 128, 8 at 256) run as row tiles
    while True:
        G = int(rng.choice([1, 2, 3, 4, 8]))
        W = int(rng.choice([1, 1, 2, 4, 8, 16]))
        if G * W <= max_rows:
            break
    n_seq = int(rng.integers(1, 6))
    lens = []
    for _ in range(n_seq):
        kind = rng.integers(0, 4)
        L = {0: 0, 1: bs + 1, 2: int(rng.integers(1, 200)), 3: int(rng.integers(200, 3000))}[int(kind)]
        lens.append(max(L, W) if L > 0 else 0)
    return rng, fmt, hd, bs, n_kv, G, W, lens


@pytest.mark.parametrize("seed", range(60))
def test_random_shapes(seed):
    rng, fmt, hd, bs, n_kv, G, W, lens = _case(seed)
    nbs = [max(1, -(-L // bs)) for L in lens]
    n_blocks = sum(nbs) + 3
    perm = rng.permutation(n_blocks).astype(np.int32)
    table = np.full((len(lens), max(nbs)), -1, np.int32)
    at = 0
    for b, nb in enumerate(nbs):
        table[b, :nb] = perm[at:at + nb]
        at += nb
    p = Pair(fmt, n_kv, hd, bs, n_blocks, table)
    n = int(sum(lens))
    if n:
        k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
        v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
        big = rng.random((n, n_kv)) < 0.05
        k[big] *= 15.0
        v[big] *= 15.0
        seq = np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lens)])
        pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
        order = rng.permutation(n)                     # cells arrive in any order
        cuts = np.sort(rng.choice(np.arange(1, n), size=min(3, n - 1), replace=False)) if n > 1 else []
        for part in np.split(order, cuts):
            p.append(k[part], v[part], seq[part], pos[part])
        p.assert_cache_equal()
    q = rng.standard_normal((len(lens), W, n_kv * G, hd)).astype(np.float32)
    ctx = np.array(lens, np.int32)
    # empty sequences (and query tokens without a visible cell) give zeros
    p.check_decode(q, ctx, workloads.sm_scale_for(hd), max_ctx=int(table.shape[1] * bs))
    for b, L in enumerate(lens):
        if L:
            p.check_compact(b, L)
            break

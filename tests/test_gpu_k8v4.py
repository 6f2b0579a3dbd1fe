"""GPU parity of the K8V4 format (int8 K, rotated 4-bit V) against the oracle.

#711 kv: --kv k8v4 streams with --kv-resident, "What": INT8 K + rotated Q4_0
V.  The append must store the oracle's codes and scales bit for bit: rows
are built in the rotated basis (y chosen, x = H y / n, so the fp32 rotation
is exact and every decision is known) to hit the cases where a careless
kernel would differ -- ties of magnitude between +m and -m (the first one
wins), quotients exactly on a half-integer (round half to even) or one to
three fp32 ulps away from one, zero blocks (scale -0, codes 8), values past
the +7 end of the code range, and the nibble order.  Decode attention and
compaction are compared on random rows at the shapes of both kernels.
"""
import numpy as np
import pytest
import torch
from scipy.linalg import hadamard

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


def _designed_rows(n, hd, rng):
    """Rows y in the rotated basis whose Q4_0 decisions sit on the edges."""
    y = np.zeros((n, hd), np.float64)
    for r in range(n):
        for b0 in range(0, hd, 32):
            kind = (r + b0 // 32) % 5
            d = float(rng.choice([1.0, 0.5, 0.25, 2.0]))     # the block's |scale|
            blk = rng.integers(-7, 8, 32) * d
            if kind == 0:     # rounding ties: y / d on half-integers
                blk = (rng.integers(-7, 7, 32) + 0.5) * d
            elif kind == 1:   # magnitude tie between +m and -m: the first wins
                blk = rng.integers(-7, 8, 32) * d
                i, j = rng.choice(32, 2, replace=False)
                blk[min(i, j)], blk[max(i, j)] = 8 * d, -8 * d
            elif kind == 2:   # zero block
                blk[:] = 0.0
            elif kind == 3:   # past +7: clamped
                blk = rng.integers(-8, 8, 32) * d
                blk[rng.integers(32)] = -8 * d
                blk[blk > 0] = 7.75 * d
            y[r, b0:b0 + 32] = blk
            if kind != 2:
                y[r, b0 + rng.integers(32)] = 8 * d * (1 if rng.random() < 0.5 else -1)
    x = (y @ hadamard(hd).T / hd).astype(np.float32)
    return x


@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("n", [96, 2100])       # a few rows, and the bulk kernel shape
def test_append_bit_exact_on_designed_rows(hd, n):
    rng = np.random.default_rng(hd + n)
    n_kv, bs = 2, 16
    v = _designed_rows(n * n_kv, hd, rng).reshape(n, n_kv, hd)
    # near-ties: nudge some values 1-3 fp32 ulps (the rotation of x is then
    # inexact, so the quotient lands a few ulps off the half-integer)
    k = v[::-1].copy()
    nudged = v.copy()
    steps = rng.integers(-3, 4, size=v.shape)
    for s in (1, 2, 3):
        nudged[steps >= s] = np.nextafter(nudged[steps >= s], np.float32(np.inf))
        nudged[steps <= -s] = np.nextafter(nudged[steps <= -s], np.float32(-np.inf))
    nb = -(-2 * n // bs)
    table = np.arange(nb, dtype=np.int32)[None]
    p = Pair("k8v4", n_kv, hd, bs, nb, table)
    p.append(k, v, np.zeros(n, np.int32), np.arange(n, dtype=np.int32))
    p.append(k, nudged, np.zeros(n, np.int32), np.arange(n, 2 * n, dtype=np.int32))
    p.assert_cache_equal()


@pytest.mark.parametrize("n_tok", [1, 3, 40, 5000])
def test_append_sizes_bit_exact(n_tok):
    rng = np.random.default_rng(n_tok)
    n_kv, hd, bs = 2, 256, 64
    nb = -(-n_tok // bs) + 1
    table = rng.permutation(nb).astype(np.int32)[None]
    k = rng.standard_normal((n_tok, n_kv, hd)).astype(np.float32)
    v = (rng.standard_normal((n_tok, n_kv, hd)) * rng.uniform(1e-3, 30, (n_tok, n_kv, 1))).astype(
        np.float32)
    p = Pair("k8v4", n_kv, hd, bs, nb, table)
    p.append(k, v, np.zeros(n_tok, np.int32), np.arange(n_tok, dtype=np.int32))
    p.assert_cache_equal()


@pytest.mark.parametrize("hd,G,W,lens", [
    (256, 4, 1, [1, 63, 64, 65, 4096]),      # the tensor-core kernel, 8-row tiles
    (256, 2, 4, [4, 300, 1025]),             # 8 rows at HD 256
    (256, 8, 1, [16, 200, 2049]),
    (128, 8, 2, [2, 777, 3000]),             # 16-row tiles
    (64, 4, 8, [8, 100, 5000]),              # 32-row tiles
    (64, 1, 1, [1, 2, 3, 4, 5]),
])
def test_decode_and_compaction(hd, G, W, lens):
    rng = np.random.default_rng(hd + G + W)
    n_kv, bs = 2, 32
    nbs = [-(-L // bs) for L in lens]
    perm = rng.permutation(sum(nbs)).astype(np.int32)
    table = np.full((len(lens), max(nbs)), -1, np.int32)
    at = 0
    for b, nb in enumerate(nbs):
        table[b, :nb] = perm[at:at + nb]
        at += nb
    p = Pair("k8v4", n_kv, hd, bs, sum(nbs), table)
    n = sum(lens)
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v[rng.random((n, n_kv)) < 0.03] *= 20.0
    seq = np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    p.append(k, v, seq, pos)
    p.assert_cache_equal()
    q = rng.standard_normal((len(lens), W, n_kv * G, hd)).astype(np.float32)
    p.check_decode(q, lens, workloads.sm_scale_for(hd))
    p.check_compact(len(lens) - 1, lens[-1])

"""GPU: gather / scatter of a sequence's cells and the cache file round trip.

kvq_gather_cells must return, bit for bit, what the oracle's gather returns
from its own pool fed the same appends; a scatter into another pool under
another block table must restore the cells exactly (gathering them again
gives the same bits, and decode attention over the restored pool equals
the original's bit for bit); save_sequence / load_sequence must do the
same through a file.  int8 codes never move without their scales (Path F
format v3: persist per-head INT8 KV scales for INT8 + persistent KV
interop, "Why").
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_kv_cache_append_gb300 as kvq
from quantized_kv_cache_append_gb300 import persist
from quantized_kv_cache_append_gb300.pool import PagedPool, row_layout
from tests.gpu_pairs import Pair, dev, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("the GPU suite needs a CUDA device")
    kvq.build()
    kvq.load_library()


def _case(fmt, n, n_kv, hd, bs, seed):
    rng = np.random.default_rng(seed)
    nb = -(-n // bs)
    table = rng.permutation(nb + 2)[:nb].astype(np.int32)[None]
    p = Pair(fmt, n_kv, hd, bs, nb + 2, table)
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    p.append(k, v, np.zeros(n, np.int32), np.arange(n, dtype=np.int32))
    return p, table


def _gather_gpu(pool, row, n):
    kdt, kn, vdt, vn, kng, vng = row_layout(pool.fmt, pool.head_dim)
    ck = torch.empty((n, pool.n_kv, kn), dtype=kdt, device="cuda")
    cv = torch.empty((n, pool.n_kv, vn), dtype=vdt, device="cuda")
    sk = sv = None
    if kng:
        sk = torch.empty((n, pool.n_kv, kng), dtype=torch.float16, device="cuda")
        sv = torch.empty((n, pool.n_kv, vng), dtype=torch.float16, device="cuda")
    assert kvq.kvq_gather_cells(pool.cache, row, n, ck, cv, sk, sv) == kvq.KVQ_OK
    torch.cuda.synchronize()
    return ck, cv, sk, sv


@pytest.mark.parametrize("fmt,hd,bs", [("f16", 128, 16), ("q8", 128, 256), ("q8", 256, 32),
                                        ("f16", 64, 64), ("k8v4", 256, 16), ("k8v4", 128, 64),
                                        ("k8v4", 64, 32)])
def test_gather_matches_oracle_and_scatter_restores(fmt, hd, bs):
    n, n_kv = 300, 2
    p, table = _case(fmt, n, n_kv, hd, bs, 40 + hd + bs)
    row = dev(table[0])
    got = _gather_gpu(p.gpu, row, n)
    ref = oracle.gather_cells(p.img, table[0], n)
    for g, r in zip(got, ref):
        if r is None:
            assert g is None
        else:
            np.testing.assert_array_equal(host_bits(g), r)
    # scatter into a second pool, other block layout
    nb = table.shape[1]
    rng = np.random.default_rng(9)
    other = rng.permutation(nb + 5)[:nb].astype(np.int32)[None]
    q2 = PagedPool(p.gpu.fmt, n_kv, hd, bs, nb + 5)
    assert kvq.kvq_scatter_cells(q2.cache, dev(other[0]), n, *got) == kvq.KVQ_OK
    back = _gather_gpu(q2, dev(other[0]), n)
    for g, b in zip(got, back):
        if g is not None:
            assert torch.equal(g, b)
    q = dev(rng.standard_normal((1, 1, 4 * n_kv, hd)).astype(np.float32))
    ctx = dev(np.array([n], np.int32))
    sm = float(1.0 / np.sqrt(hd))
    o1 = p.gpu.decode(q, ctx, n, p.bt, sm)
    o2 = q2.decode(q, ctx, n, dev(other), sm)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("fmt", ["f16", "q8", "k8v4"])
def test_file_round_trip(tmp_path, fmt):
    n, n_kv, hd, bs = 200, 4, 128, 64
    p, table = _case(fmt, n, n_kv, hd, bs, 50)
    path = tmp_path / "seq.kvq"
    tokens = np.arange(7, 7 + n, dtype=np.int32)
    persist.save_sequence(path, p.gpu, dev(table[0]), n, tokens)
    nb = table.shape[1]
    other = np.arange(nb, dtype=np.int32)[None]
    fresh = PagedPool(p.gpu.fmt, n_kv, hd, bs, nb)
    n2, t2 = persist.load_sequence(path, fresh, dev(other[0]))
    assert n2 == n and np.array_equal(t2, tokens)
    a = _gather_gpu(p.gpu, dev(table[0]), n)
    b = _gather_gpu(fresh, dev(other[0]), n)
    for x, y in zip(a, b):
        if x is not None:
            assert torch.equal(x, y)


def test_int8_without_scales_is_refused():
    p, table = _case("q8", 32, 1, 64, 16, 60)
    row = dev(table[0])
    ck = torch.empty((32, 1, 64), dtype=torch.int8, device="cuda")
    cv = torch.empty_like(ck)
    assert kvq.kvq_gather_cells(p.gpu.cache, row, 32, ck, cv, None, None) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_scatter_cells(p.gpu.cache, row, 32, ck, cv, None, None) == kvq.KVQ_ERR_ARG
    torch.cuda.synchronize()

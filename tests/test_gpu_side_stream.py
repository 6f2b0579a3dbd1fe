"""GPU: every call driven through the package on a stream other than
torch's current one (a torch stream, and the same stream as a raw handle)
gives the bits the current stream gives, and the tensors the package
allocates for such a call (outputs, workspace, staging of ids and of a
restored sequence) belong to that stream.

The library runs each call on the stream it is given; these tests make the
Python side keep its own copies and allocations on that stream too.
"""
import numpy as np
import pytest
import torch

import quantized_kv_cache_append_gb300 as kvq
from quantized_kv_cache_append_gb300 import persist
from quantized_kv_cache_append_gb300.pool import PagedPool
from quantized_kv_cache_append_gb300.stream import StreamedPool
from tests.gpu_pairs import FORMATS, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("the GPU suite needs a CUDA device")
    kvq.build()
    kvq.load_library()


def _filled_pool(fmt, n, n_kv, hd, bs, seed):
    rng = np.random.default_rng(seed)
    nb = -(-n // bs)
    table = rng.permutation(nb + 3)[:nb].astype(np.int32)[None]
    pool = PagedPool(FORMATS[fmt][0], n_kv, hd, bs, nb + 3)
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    pool.append(dev(k), dev(v), dev(np.zeros(n, np.int32)), dev(np.arange(n, dtype=np.int32)),
                dev(table))
    return pool, table, rng


@pytest.mark.parametrize("fmt", ["f16", "q8", "k8v4"])
def test_decode_and_compaction_on_a_side_stream(fmt):
    n, n_kv, hd, bs = 700, 2, 128, 64
    pool, table, rng = _filled_pool(fmt, n, n_kv, hd, bs, 70 + len(fmt))
    bt = dev(table)
    q = dev(rng.standard_normal((1, 1, 4 * n_kv, hd)).astype(np.float32))
    ctx = dev(np.array([n], np.int32))
    sm = float(1.0 / np.sqrt(hd))
    ref = pool.decode(q, ctx, n, bt, sm)
    ref_k, ref_v = pool.compact(bt[0], n)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for s in (side, side.cuda_stream):
        out = pool.decode(q, ctx, n, bt, sm, stream=s)
        ck, cv = pool.compact(bt[0], n, stream=s)
        side.synchronize()
        assert torch.equal(out, ref)
        assert torch.equal(ck, ref_k) and torch.equal(cv, ref_v)


@pytest.mark.parametrize("fmt", ["q8", "k8v4"])
def test_fetch_on_a_side_stream(fmt):
    n_kv, hd, bs, n_host, n_slots = 2, 128, 16, 24, 8
    rng = np.random.default_rng(80)
    sp = StreamedPool(FORMATS[fmt][0], n_kv, hd, bs, n_host, n_slots)
    n = n_host * bs
    table = np.arange(n_host, dtype=np.int32)[None]
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    sp.append_host(dev(k), dev(v), dev(np.zeros(n, np.int32)), dev(np.arange(n, dtype=np.int32)),
                   dev(table))
    torch.cuda.synchronize()
    row = rng.permutation(n_host)[:n_slots].astype(np.int32)[None]
    slots, src, dst, hits = sp.plan(row, np.array([n_slots * bs], np.int32))
    assert hits == 0 and len(src) == n_slots
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    sp.fetch(src, dst, stream=side)
    side.synchronize()
    for b, s in zip(src.tolist(), dst.tolist()):
        assert torch.equal(sp.window.k[s].cpu(), sp.host.k[b])
        assert torch.equal(sp.window.v[s].cpu(), sp.host.v[b])
        assert torch.equal(sp.window.ks[s].cpu(), sp.host.ks[b])
        assert torch.equal(sp.window.vs[s].cpu(), sp.host.vs[b])


@pytest.mark.parametrize("fmt", ["f16", "k8v4"])
def test_sequence_file_on_a_side_stream(tmp_path, fmt):
    n, n_kv, hd, bs = 300, 2, 128, 32
    pool, table, _ = _filled_pool(fmt, n, n_kv, hd, bs, 90)
    path = tmp_path / "seq.kvq"
    row = dev(table[0])
    nb = table.shape[1]
    fresh = PagedPool(pool.fmt, n_kv, hd, bs, nb)
    other = dev(np.arange(nb, dtype=np.int32))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())   # everything above is in place
    persist.save_sequence(path, pool, row, n, stream=side)
    n2, _ = persist.load_sequence(path, fresh, other, stream=side.cuda_stream)
    assert n2 == n
    a_k, a_v = pool.compact(row, n)
    b_k, b_v = fresh.compact(other, n)
    torch.cuda.synchronize()
    assert torch.equal(a_k, b_k) and torch.equal(a_v, b_v)

"""GPU: the streamed pool (host copy + resident window) against a fully
resident pool.

#711 kv: --kv k8v4 streams with --kv-resident, "Tests": streamed and
resident attention are bitwise equal, in every format.  Here a batch of
sequences grows step by step; each step appends to the host copy (and to a
resident pool and the oracle image), plans the window, fetches the missing
blocks from the host copy, appends to the window under the slot table, and
decodes: the window's attention must equal the resident pool's bit for
bit (same bytes, same kernels, other block ids), its compaction too, the
window must miss and hit, and the host copy must hold the oracle's bits.
"""
import numpy as np
import pytest
import torch

import quantized_kv_cache_append_gb300 as kvq
from quantized_kv_cache_append_gb300.stream import StreamedPool
from tests.gpu_pairs import FORMATS, Pair, dev, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("the GPU suite needs a CUDA device")
    kvq.build()
    kvq.load_library()


@pytest.mark.parametrize("fmt,hd", [("f16", 128), ("q8", 128), ("k8v4", 256), ("q8", 64)])
def test_streamed_attention_is_bitwise_the_resident_attention(fmt, hd):
    rng = np.random.default_rng(hd + len(fmt))
    n_kv, G, bs = 2, 4, 16
    n_seq, max_blocks = 6, 12
    n_host = n_seq * max_blocks + 3
    n_slots = 2 * max_blocks            # two sequences of a batch always fit
    table = rng.permutation(n_host)[: n_seq * max_blocks].astype(np.int32).reshape(n_seq, max_blocks)
    sp = StreamedPool(FORMATS[fmt][0], n_kv, hd, bs, n_host, n_slots)
    ref = Pair(fmt, n_kv, hd, bs, n_host, table)
    lens = np.zeros(n_seq, np.int32)
    d_table = dev(table)
    sm = float(1.0 / np.sqrt(hd))
    fetched = hits = 0
    for step in range(36):
        batch = np.sort(rng.choice(n_seq, size=2, replace=False))
        room = max_blocks * bs - lens[batch]
        new = np.minimum(rng.integers(1, 40, 2), room)
        if new.sum() == 0:
            continue
        seq_full = np.concatenate([np.full(n, b, np.int32) for b, n in zip(batch, new)])
        seq_rel = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(new)])
        pos = np.concatenate([np.arange(lens[b], lens[b] + n, dtype=np.int32)
                              for b, n in zip(batch, new)])
        k = rng.standard_normal((len(pos), n_kv, hd)).astype(np.float32)
        v = rng.standard_normal((len(pos), n_kv, hd)).astype(np.float32)
        lens[batch] += new
        ref.append(k, v, seq_full, pos)
        dk, dv, dpos = dev(k), dev(v), dev(pos)
        sp.append_host(dk, dv, dev(seq_full), dpos, d_table)
        ctx = lens[batch].copy()
        slot_table, src, dst, h = sp.plan(table[batch], ctx)
        sp.fetch(src, dst)
        d_slots = dev(slot_table)
        sp.window.append(dk, dv, dev(seq_rel), dpos, d_slots)
        fetched += len(src)
        hits += h
        q = dev(rng.standard_normal((2, 1, n_kv * G, hd)).astype(np.float32))
        max_ctx = max_blocks * bs
        out_w = sp.window.decode(q, dev(ctx), max_ctx, d_slots, sm)
        out_r = ref.gpu.decode(q, dev(ctx), max_ctx, dev(table[batch]), sm)
        torch.cuda.synchronize()
        assert torch.equal(out_w, out_r), f"step {step}: streamed attention differs"
        if step % 9 == 8:
            cw = sp.window.compact(d_slots[0], int(ctx[0]))
            cr = ref.gpu.compact(dev(table[batch[0]]), int(ctx[0]))
            torch.cuda.synchronize()
            assert all(torch.equal(a, b) for a, b in zip(cw, cr))
    assert fetched > n_slots and hits > 0           # the window both missed and hit
    # the host copy holds the resident pool's (and so the oracle's) bits
    torch.cuda.synchronize()
    ref.assert_cache_equal()
    for name in ("k", "v", "ks", "vs"):
        a, b = getattr(sp.host, name), getattr(ref.gpu, name)
        if a is not None:
            assert np.array_equal(host_bits(a), host_bits(b)), f"host copy {name} differs"


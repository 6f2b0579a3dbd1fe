"""GPU: the failure path of the decode's and the chunk attention's bounded waits.

Refuse rather than return silent garbage (#711 kv: --kv k8v4 streams with
--kv-resident, "How" and "Tests"; Path F format v3, "Why"): every wait of
the tensor-core decode for a copy into shared memory is bounded, and a
wait that runs out turns the affected output rows into NaN instead of
hanging or returning a wrong number.  kvq_decode_attn_lost_wait_test makes
every wait run out (each copy stage expects 16 bytes that no copy sends,
waits bounded to a few thousand polls): the call must return KVQ_OK with
NaN rows, and the context must stay usable -- the next ordinary decode on
the same pool is correct.  kvq_chunk_attn_lost_wait_test does the same for
the prompt-chunk attention (every K and V stage short of 16 bytes): NaN in
every output row, on an unsplit grid and through the distributed-shared-
memory merge of a short chunk's key splits, then a correct ordinary call.
No fault, trap or unbounded wait is involved.
"""
import numpy as np
import pytest
import torch

import workloads
import quantized_kv_cache_append_gb300 as kvq
from tests.gpu_pairs import Pair, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("the GPU suite needs a CUDA device")
    kvq.build()
    kvq.load_library()


@pytest.mark.parametrize("fmt", ["f16", "q8", "k8v4"])
def test_lost_copy_waits_give_nan_rows_and_leave_the_context_usable(fmt):
    wl = workloads.make("tiny")
    p = Pair(fmt, wl.n_kv, wl.head_dim, wl.block_size, wl.n_blocks, wl.block_table)
    p.append(wl.k, wl.v, wl.tok_seq, wl.tok_pos)
    n_seq, W, n_q, hd = wl.q.shape
    L = int(wl.ctx_lens[0])
    q, ctx = dev(wl.q), dev(wl.ctx_lens)
    out = torch.zeros(wl.q.shape, dtype=torch.float32, device="cuda")
    ws_bytes = p.gpu.workspace_bytes(n_seq, W, n_q, L)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = kvq.kvq_decode_attn_lost_wait_test(p.gpu.cache, q, n_seq, W, n_q, ctx, L, p.bt,
                                            p.bt_host.shape[1], wl.sm_scale, out, ws, ws_bytes,
                                            4096, 16)
    assert st == kvq.KVQ_OK, kvq.kvq_status_string(st)
    torch.cuda.synchronize()                       # no CUDA error: the context is intact
    assert torch.isnan(out).all(), "a lost copy wait must give NaN rows"
    # the next ordinary call on the same pool and workspace is correct
    p.check_decode(wl.q, wl.ctx_lens, wl.sm_scale)


@pytest.mark.parametrize("hd,n_kv,G,P,T", [
    (64, 8, 4, 700, 640),      # 160 (row tile, KV head) CTAs: no key split
    (128, 2, 4, 8192, 64),     # a short chunk: key tiles split over clusters, merged in DSMEM
    (256, 1, 2, 3000, 100),
])
def test_chunk_lost_waits_give_nan_rows_and_leave_the_context_usable(hd, n_kv, G, P, T):
    # kvq_chunk_attn_lost_wait_test: every K and V stage expects 16 bytes
    # that no copy sends and every wait is bounded to 4096 polls, so every
    # role's wait runs out; the rows must come back NaN (through the merge
    # of the key splits as well), with no CUDA error, and the next ordinary
    # call must be correct
    import oracle
    from tests.gpu_pairs import assert_attention_close
    rng = np.random.default_rng(900 + hd)
    k16 = oracle.fp16_bits(rng.standard_normal((n_kv, P, hd)).astype(np.float32))
    v16 = oracle.fp16_bits(rng.standard_normal((n_kv, P, hd)).astype(np.float32))
    q = rng.standard_normal((T, n_kv * G, hd)).astype(np.float32)
    kd = dev(k16.view(np.int16)).view(torch.float16)
    vd = dev(v16.view(np.int16)).view(torch.float16)
    qd = dev(q)
    sm = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    out = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    st = kvq.kvq_chunk_attn_lost_wait_test(kd, vd, n_kv, P, hd, qd, T, n_kv * G, sm, out, 4096, 16)
    assert st == kvq.KVQ_OK, kvq.kvq_status_string(st)
    torch.cuda.synchronize()                       # no CUDA error: the context is intact
    assert torch.isnan(out).all(), "a lost wait must give NaN rows"
    st = kvq.kvq_chunk_attn(kd, vd, n_kv, P, hd, qd, T, n_kv * G, sm, out)
    assert st == kvq.KVQ_OK, kvq.kvq_status_string(st)
    torch.cuda.synchronize()
    assert_attention_close(out.cpu().numpy(), oracle.chunk_attention(k16, v16, q, sm))


def test_chunk_lost_wait_test_refuses_bad_knobs():
    k = torch.zeros(1, 64, 128, dtype=torch.float16, device="cuda")
    q = torch.zeros(4, 4, 128, device="cuda")
    out = torch.zeros_like(q)
    call = lambda limit, extra: kvq.kvq_chunk_attn_lost_wait_test(k, k, 1, 64, 128, q, 4, 4, 0.1,
                                                                  out, limit, extra)
    assert call(0, 16) == kvq.KVQ_ERR_ARG
    assert call(4096, 0) == kvq.KVQ_ERR_ARG
    assert call(4096, 24) == kvq.KVQ_ERR_ARG         # not a multiple of 16
    assert call((1 << 25) + 1, 16) == kvq.KVQ_ERR_ARG
    torch.cuda.synchronize()


def test_lost_wait_test_refuses_bad_knobs():
    wl = workloads.make("tiny")
    p = Pair("q8", wl.n_kv, wl.head_dim, wl.block_size, wl.n_blocks, wl.block_table)
    n_seq, W, n_q, hd = wl.q.shape
    L = int(wl.ctx_lens[0])
    q, ctx = dev(wl.q), dev(wl.ctx_lens)
    out = torch.zeros(wl.q.shape, dtype=torch.float32, device="cuda")
    ws_bytes = p.gpu.workspace_bytes(n_seq, W, n_q, L)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    call = lambda limit, extra: kvq.kvq_decode_attn_lost_wait_test(
        p.gpu.cache, q, n_seq, W, n_q, ctx, L, p.bt, p.bt_host.shape[1], wl.sm_scale, out, ws,
        ws_bytes, limit, extra)
    assert call(0, 16) == kvq.KVQ_ERR_ARG
    assert call(4096, 0) == kvq.KVQ_ERR_ARG
    assert call(4096, 8) == kvq.KVQ_ERR_ARG          # not a multiple of 16
    assert call((1 << 25) + 1, 16) == kvq.KVQ_ERR_ARG
    torch.cuda.synchronize()

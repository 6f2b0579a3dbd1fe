"""kvq_decode_attn_static: decode attention for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc at the point where they
decode: code that runs while a CUDA graph is being captured (allocation is
not allowed during capture), a plugin inside a framework whose caching
allocator owns the device memory, or a real-time loop whose memory was
fixed at start-up.  kvq_decode_attn_static serves them with scratch that
the library keeps in a device array of its own.

This file checks, through the C ABI, that it returns what kvq_decode_attn
(with a caller-provided workspace) returns, on two calls in a row with
different shapes (the second call finds the first call's leftovers in the
shared scratch), that a request whose full split plan does not fit the
array is cut into fewer splits and still matches the float64 oracle, and
that a request too large even with one split per (sequence, KV head) is
refused before anything runs.  It is collected last so that a run stopping at the
first failure has run every other test first; it also passes on its own.
"""
import numpy as np
import pytest
import torch

import quantized_kv_cache_append_gb300 as kvq
from quantized_kv_cache_append_gb300.pool import PagedPool

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-3
REL_L2 = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    kvq.build()
    kvq.load_library()


def _case(fmt, n_seq, n_kv, G, W, hd, bs, lens, seed):
    g = torch.Generator().manual_seed(seed)
    nbs = [-(-L // bs) for L in lens]
    n_blocks = sum(nbs)
    perm = torch.randperm(n_blocks, generator=g).to(torch.int32)
    table = torch.full((n_seq, max(nbs)), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(nbs):
        table[b, :n] = perm[at:at + n]
        at += n
    n_tok = sum(lens)
    k = torch.randn(n_tok, n_kv, hd, generator=g)
    v = torch.randn(n_tok, n_kv, hd, generator=g)
    seq = torch.cat([torch.full((L,), b, dtype=torch.int32) for b, L in enumerate(lens)])
    pos = torch.cat([torch.arange(L, dtype=torch.int32) for L in lens])
    q = torch.randn(n_seq, W, n_kv * G, hd, generator=g)
    pool = PagedPool(fmt, n_kv, hd, bs, n_blocks)
    bt = table.cuda()
    pool.append(k.cuda(), v.cuda(), seq.cuda(), pos.cuda(), bt)
    return pool, q.cuda(), torch.tensor(lens, dtype=torch.int32).cuda(), bt


def _static(pool, q, ctx, max_ctx, bt, sm):
    n_seq, W, n_q, _ = q.shape
    out = torch.full_like(q, float("nan"))
    st = kvq.kvq_decode_attn_static(pool.cache, q, n_seq, W, n_q, ctx, max_ctx, bt,
                                    bt.shape[1], sm, out)
    assert st == kvq.KVQ_OK, kvq.kvq_status_string(st)
    return out


def _with_workspace(pool, q, ctx, max_ctx, bt, sm):
    n_seq, W, n_q, _ = q.shape
    out = torch.full_like(q, float("nan"))
    need = kvq.kvq_decode_workspace_bytes(pool.cache, n_seq, W, n_q, max_ctx)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    st = kvq.kvq_decode_attn(pool.cache, q, n_seq, W, n_q, ctx, max_ctx, bt, bt.shape[1], sm,
                             out, ws, need)
    assert st == kvq.KVQ_OK, kvq.kvq_status_string(st)
    return out


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    assert np.isfinite(a).all() and np.isfinite(b).all()
    d = a - b
    assert np.abs(d).max() <= MAX_ABS
    assert np.linalg.norm(d) <= REL_L2 * np.linalg.norm(b)


def test_static_scratch_matches_workspace_entry_point_twice_in_a_row():
    cases = [
        # int8 cache, GQA 32/8, head_dim 128, ragged batch
        dict(fmt=kvq.KVQ_Q8, n_seq=3, n_kv=8, G=4, W=1, hd=128, bs=256,
             lens=[4096, 1500, 333], seed=1),
        # FP16 cache, 16/2 heads, head_dim 256, a 2-token verify window
        dict(fmt=kvq.KVQ_F16, n_seq=1, n_kv=2, G=4, W=2, hd=256, bs=64,
             lens=[20000], seed=2),
    ]
    for c in cases:
        pool, q, ctx, bt = _case(c["fmt"], c["n_seq"], c["n_kv"], c["G"], c["W"], c["hd"],
                                 c["bs"], c["lens"], c["seed"])
        sm = float(1.0 / np.sqrt(c["hd"]))
        max_ctx = max(c["lens"])
        got = _static(pool, q, ctx, max_ctx, bt, sm)
        ref = _with_workspace(pool, q, ctx, max_ctx, bt, sm)
        torch.cuda.synchronize()
        _close(got, ref)


def test_request_beyond_the_static_scratch_is_refused():
    # 256 sequences x 8 KV heads x 16 rows x 128 dims of fp32 partials is
    # 16 MiB, more than the 8 MiB array: refused before any launch (every
    # buffer below is still valid, so nothing could go out of bounds).
    n_seq, n_kv, G, W, hd, bs = 256, 8, 4, 4, 128, 16
    pool = PagedPool(kvq.KVQ_Q8, n_kv, hd, bs, n_seq * 4)
    bt = torch.arange(n_seq * 4, dtype=torch.int32, device="cuda").view(n_seq, 4)
    q = torch.zeros(n_seq, W, n_kv * G, hd, device="cuda")
    out = torch.zeros_like(q)
    ctx = torch.full((n_seq,), 64, dtype=torch.int32, device="cuda")
    need = kvq.kvq_decode_workspace_bytes(pool.cache, n_seq, W, n_kv * G, 64)
    assert need > kvq.KVQ_STATIC_SCRATCH_BYTES
    st = kvq.kvq_decode_attn_static(pool.cache, q, n_seq, W, n_kv * G, ctx, 64, bt, 4,
                                    0.1, out)
    assert st == kvq.KVQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not out.any()


def test_plan_lowered_to_fit_the_static_scratch_matches_the_oracle():
    # A verify window of 4 tokens on 32 ragged int8 sequences: the full split
    # plan needs more partials than the 8 MiB array holds, so the call cuts
    # the context into fewer splits until they fit.  Its output must still be
    # the attention the pages define (the float64 oracle on its own cache,
    # fed the same cells; same bar as every other decode) and agree with the
    # workspace entry point.
    import oracle
    from tests.gpu_pairs import Pair, assert_attention_close, dev

    n_seq, n_kv, G, W, hd, bs = 32, 8, 4, 4, 128, 256
    rng = np.random.default_rng(5)
    lens = rng.integers(1024, 8193, n_seq).astype(np.int32)
    max_ctx = int(lens.max())
    nbs = [-(-int(L) // bs) for L in lens]
    perm = rng.permutation(sum(nbs)).astype(np.int32)
    table = np.full((n_seq, max(nbs)), -1, np.int32)
    at = 0
    for b, n in enumerate(nbs):
        table[b, :n] = perm[at:at + n]
        at += n
    pair = Pair("q8", n_kv, hd, bs, sum(nbs), table)
    n_tok = int(lens.sum())
    k = rng.standard_normal((n_tok, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n_tok, n_kv, hd)).astype(np.float32)
    seq = np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    pair.append(k, v, seq, pos)
    q = rng.standard_normal((n_seq, W, n_kv * G, hd)).astype(np.float32)
    sm = float(np.float32(1.0) / np.sqrt(np.float32(hd)))

    pool = pair.gpu
    need = kvq.kvq_decode_workspace_bytes(pool.cache, n_seq, W, n_kv * G, max_ctx)
    assert need > kvq.KVQ_STATIC_SCRATCH_BYTES
    qd, ctx = dev(q), dev(lens)
    got = _static(pool, qd, ctx, max_ctx, pair.bt, sm)
    ref = _with_workspace(pool, qd, ctx, max_ctx, pair.bt, sm)
    torch.cuda.synchronize()
    _close(got, ref)

    path = oracle.parallel_library(8)   # the same oracle on 8 threads (bitwise equal)
    if path is not None:
        with oracle.use_library(path):
            want = pair.decode_oracle(q, lens, sm)
    else:
        want = pair.decode_oracle(q, lens, sm)
    assert_attention_close(got.cpu().numpy(), want)

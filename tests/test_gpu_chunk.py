"""GPU parity of the prompt-chunk attention (kvq_chunk_attn) against the
oracle's float64 chunk attention over the same fp16 staging.

The staging is what compaction writes for the chunk's sequence (#3084
qwen35: FP16 K/V cache by default, int8 with --kv-q8, "Extra Notes": the
prompt chunk's Q K^T and P V products read it).  Small shapes compare every
output with the oracle, which builds its own staging from its own pool;
the full chunk (131072 cells, a 4096-token chunk, 32/8 heads, head_dim 128)
compares sampled tokens, each an oracle call over exactly the cells that
token sees.  Bars: max-abs 2e-3 and relative L2 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_kv_cache_append_gb300 as kvq
from tests.gpu_pairs import assert_attention_close, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("the GPU suite needs a CUDA device")
    kvq.build()
    kvq.load_library()


def _sm(hd):
    return float(np.float32(1.0) / np.sqrt(np.float32(hd)))


def _staging_from_oracle_pool(fmt, n_kv, hd, P, seed):
    """An oracle pool of P cells (shuffled blocks of 16), compacted by the
    oracle: fp16 bits [n_kv][P][hd] for K and V."""
    rng = np.random.default_rng(seed)
    bs = 16
    nb = -(-P // bs)
    table = rng.permutation(nb).astype(np.int32)[None]
    k = rng.standard_normal((P, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((P, n_kv, hd)).astype(np.float32)
    k[:, :, rng.integers(0, hd, 4)] *= 20.0          # outlier channels
    pool = oracle.PoolImage(fmt, n_kv, hd, bs, nb)
    oracle.append(pool, k, v, np.zeros(P, np.int32), np.arange(P, dtype=np.int32), table)
    return oracle.compact_f16(pool, table[0], P)


def _gpu_chunk(k16, v16, q, sm):
    n_kv, P, hd = k16.shape
    T, n_q, _ = q.shape
    kd = dev(k16.view(np.int16)).view(torch.float16)
    vd = dev(v16.view(np.int16)).view(torch.float16)
    qd = dev(q)
    out = torch.full(q.shape, float("nan"), device="cuda")
    st = kvq.kvq_chunk_attn(kd, vd, n_kv, P, hd, qd, T, n_q, sm, out)
    assert st == kvq.KVQ_OK, kvq.kvq_status_string(st)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("fmt,n_kv,G,hd,P,T", [
    (oracle.FMT_F16, 2, 4, 128, 1000, 128),
    (oracle.FMT_Q8, 2, 4, 128, 1000, 128),
    (oracle.FMT_F16, 1, 8, 64, 300, 300),      # the whole prompt is the chunk
    (oracle.FMT_Q8, 2, 2, 256, 520, 65),       # ragged row and key tiles
    (oracle.FMT_F16, 4, 1, 128, 64, 1),        # one token, one key tile
    (oracle.FMT_Q8, 1, 4, 128, 2048, 256),
    (oracle.FMT_F16, 3, 3, 64, 777, 40),       # G = 3: rows of a tile span tokens unevenly
    (oracle.FMT_K8V4, 2, 4, 128, 1000, 128),   # staging of a K8V4 cache (V rotated back)
    (oracle.FMT_F16, 2, 4, 64, 4096, 512),     # head_dim 64 on tensor memory: many key and row tiles
    (oracle.FMT_Q8, 3, 2, 64, 1500, 700),      # head_dim 64, ragged tiles, rows spanning tokens
    (oracle.FMT_F16, 2, 4, 256, 2000, 400),    # head_dim 256: 64-key tiles, one V stage, many tiles
    (oracle.FMT_K8V4, 1, 3, 256, 900, 333),    # head_dim 256, G = 3, ragged key and row tiles
    # short chunks over long contexts: few row tiles, so the key tiles are
    # split over a cluster of CTAs that merge through distributed shared memory
    (oracle.FMT_F16, 2, 4, 128, 8192, 64),
    (oracle.FMT_Q8, 1, 8, 64, 5000, 40),
    (oracle.FMT_K8V4, 2, 2, 256, 3000, 100),
    (oracle.FMT_F16, 1, 1, 128, 4096, 1),      # one token, one row
    # 160 (row tile, KV head) CTAs: no key split
    (oracle.FMT_F16, 8, 4, 64, 700, 640),
    (oracle.FMT_Q8, 8, 4, 256, 700, 640),
])
def test_chunk_matches_oracle(fmt, n_kv, G, hd, P, T):
    k16, v16 = _staging_from_oracle_pool(fmt, n_kv, hd, P, 31 + hd + T)
    rng = np.random.default_rng(77 + P)
    q = rng.standard_normal((T, n_kv * G, hd)).astype(np.float32)
    got = _gpu_chunk(k16, v16, q, _sm(hd))
    ref = oracle.chunk_attention(k16, v16, q, _sm(hd))
    assert_attention_close(got, ref)


def test_full_chunk_sampled_tokens():
    # the chunk_verify sizes: 126976 + 4096 cells, 32/8 heads, head_dim 128
    n_kv, G, hd, P, T = 8, 4, 128, 131072, 4096
    g = torch.Generator().manual_seed(1005)
    kf = torch.randn(n_kv, P, hd, generator=g)
    vf = torch.randn(n_kv, P, hd, generator=g)
    q = torch.randn(T, n_kv * G, hd, generator=g).numpy()
    k16 = oracle.fp16_bits(kf.numpy())
    v16 = oracle.fp16_bits(vf.numpy())
    got = _gpu_chunk(k16, v16, q, _sm(hd))
    assert np.isfinite(got).all()
    for t in (0, 1, 1023, 2048, 4095):
        n_vis = P - T + t + 1
        ref = oracle.chunk_attention(np.ascontiguousarray(k16[:, :n_vis]),
                                     np.ascontiguousarray(v16[:, :n_vis]), q[t:t + 1], _sm(hd))
        assert_attention_close(got[t:t + 1], ref)


def test_short_chunk_sampled_tokens():
    # the benchmark's short chunk: 256 tokens over 131072 cells, 32/8 heads,
    # head_dim 128 -- 64 (row tile, KV head) pairs, so the key tiles are
    # split over clusters of CTAs and merged through distributed shared
    # memory; sampled tokens against the oracle over exactly their cells
    n_kv, G, hd, P, T = 8, 4, 128, 131072, 256
    g = torch.Generator().manual_seed(1777)
    kf = torch.randn(n_kv, P, hd, generator=g)
    vf = torch.randn(n_kv, P, hd, generator=g)
    q = torch.randn(T, n_kv * G, hd, generator=g).numpy()
    k16 = oracle.fp16_bits(kf.numpy())
    v16 = oracle.fp16_bits(vf.numpy())
    got = _gpu_chunk(k16, v16, q, _sm(hd))
    assert np.isfinite(got).all()
    for t in (0, 1, 127, 128, 255):
        n_vis = P - T + t + 1
        ref = oracle.chunk_attention(np.ascontiguousarray(k16[:, :n_vis]),
                                     np.ascontiguousarray(v16[:, :n_vis]), q[t:t + 1], _sm(hd))
        assert_attention_close(got[t:t + 1], ref)


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_chunk_rising_logits(hd):
    # logits that climb along the keys (a ramp in one K channel, q aligned
    # with it): the running maximum rises past the lazy threshold every
    # couple of key tiles, so O is rescaled in tensor memory again and
    # again, each time after the previous tile's P V has completed
    n_kv, G, P, T = 2, 4, 2048, 512
    rng = np.random.default_rng(4242 + hd)
    k = rng.standard_normal((n_kv, P, hd)).astype(np.float32)
    v = rng.standard_normal((n_kv, P, hd)).astype(np.float32)
    sm = _sm(hd)
    # + 8 in the log2 domain every 256 keys
    k[:, :, 0] = np.arange(P, dtype=np.float32) * (8.0 / 256) / (sm * np.log2(np.e))
    q = rng.standard_normal((T, n_kv * G, hd)).astype(np.float32) * 0.1
    q[:, :, 0] = 1.0
    k16, v16 = oracle.fp16_bits(k), oracle.fp16_bits(v)
    got = _gpu_chunk(k16, v16, q, sm)
    ref = oracle.chunk_attention(k16, v16, q, sm)
    assert_attention_close(got, ref)


def test_chunk_refuses_bad_arguments():
    k = torch.zeros(1, 64, 128, dtype=torch.float16, device="cuda")
    q = torch.zeros(4, 4, 128, device="cuda")
    out = torch.zeros_like(q)
    ok = kvq.kvq_chunk_attn(k, k, 1, 64, 128, q, 4, 4, 0.1, out)
    assert ok == kvq.KVQ_OK
    assert kvq.kvq_chunk_attn(k, k, 1, 64, 128, q, 65, 4, 0.1, out) == kvq.KVQ_ERR_ARG   # T > P
    assert kvq.kvq_chunk_attn(k, k, 3, 64, 128, q, 4, 4, 0.1, out) == kvq.KVQ_ERR_ARG   # n_q % n_kv
    assert kvq.kvq_chunk_attn(k, k, 1, 64, 96, q, 4, 4, 0.1, out) == kvq.KVQ_ERR_UNSUPPORTED
    assert kvq.kvq_chunk_attn(None, k, 1, 64, 128, q, 4, 4, 0.1, out) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_chunk_attn(k, k, 1, 64, 128, q, 4, 4, float("nan"), out) == kvq.KVQ_ERR_ARG
    torch.cuda.synchronize()

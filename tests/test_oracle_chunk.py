"""Pins for the oracle's prompt-chunk attention over fp16 staging.

The prompt chunk's Q K^T and P V products read the contiguous [kvh][P][HD]
fp16 halves that compaction writes (#3084 qwen35: FP16 K/V cache by
default, int8 with --kv-q8, "Extra Notes"); the chunk's tokens are the
sequence's last T cells, each attending causally to every cell up to its
own.  The oracle is pinned by torch's scaled_dot_product_attention in
float64 with that mask written out, by the oracle's own paged decode
attention (a separate code path, itself pinned) over an FP16 pool holding
the same values, and by closed forms (one visible cell gives V exactly,
equal keys give the running mean of V).
"""
import numpy as np
import pytest
import torch

import oracle


def _sm(hd):
    return float(np.float32(1.0) / np.sqrt(np.float32(hd)))


def _random_staging(rng, n_kv, P, hd):
    k = oracle.fp16_bits(rng.standard_normal((n_kv, P, hd)).astype(np.float32))
    v = oracle.fp16_bits(rng.standard_normal((n_kv, P, hd)).astype(np.float32))
    return k, v


def _sdpa(k16, v16, q, sm):
    n_kv, P, hd = k16.shape
    T, n_q, _ = q.shape
    G = n_q // n_kv
    K = torch.from_numpy(oracle.fp16_value(k16).astype(np.float64)).repeat_interleave(G, 0)[None]
    V = torch.from_numpy(oracle.fp16_value(v16).astype(np.float64)).repeat_interleave(G, 0)[None]
    Q = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]   # [1][n_q][T][hd]
    mask = torch.arange(P)[None, :] <= (P - T + torch.arange(T))[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(
        Q, K, V, attn_mask=mask, scale=float(np.float64(np.float32(sm))))
    return out[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("n_kv,G,hd,P,T", [
    (1, 4, 128, 200, 37), (2, 2, 64, 96, 96), (2, 8, 256, 130, 5), (3, 1, 128, 64, 1),
])
def test_matches_torch_sdpa(n_kv, G, hd, P, T):
    rng = np.random.default_rng(100 + hd + T)
    k16, v16 = _random_staging(rng, n_kv, P, hd)
    q = rng.standard_normal((T, n_kv * G, hd)).astype(np.float32)
    out = oracle.chunk_attention(k16, v16, q, _sm(hd))
    np.testing.assert_allclose(out, _sdpa(k16, v16, q, _sm(hd)), rtol=1e-10, atol=1e-10)


def test_matches_paged_attention_over_an_fp16_pool():
    # an FP16 pool holding the staging values (fp16(x) of fp16 values is
    # exact), read by the paged decode attention with W = T
    rng = np.random.default_rng(7)
    n_kv, G, hd, P, T, bs = 2, 4, 128, 150, 12, 16
    k16, v16 = _random_staging(rng, n_kv, P, hd)
    nb = -(-P // bs)
    table = rng.permutation(nb).astype(np.int32)[None]
    pool = oracle.PoolImage(oracle.FMT_F16, n_kv, hd, bs, nb)
    kf = oracle.fp16_value(k16).astype(np.float32).transpose(1, 0, 2).copy()  # [P][n_kv][hd]
    vf = oracle.fp16_value(v16).astype(np.float32).transpose(1, 0, 2).copy()
    oracle.append(pool, kf, vf, np.zeros(P, np.int32), np.arange(P, dtype=np.int32), table)
    q = rng.standard_normal((T, n_kv * G, hd)).astype(np.float32)
    paged = oracle.attention(pool, q[None], np.array([P], np.int32), table, _sm(hd))[0]
    chunk = oracle.chunk_attention(k16, v16, q, _sm(hd))
    np.testing.assert_allclose(chunk, paged, rtol=1e-12, atol=1e-12)


def test_first_token_of_a_whole_prompt_sees_one_cell():
    # T = P: token 0 sees cell 0 only, so its output is V[0] exactly
    rng = np.random.default_rng(8)
    k16, v16 = _random_staging(rng, 2, 40, 64)
    q = rng.standard_normal((40, 4, 64)).astype(np.float32)
    out = oracle.chunk_attention(k16, v16, q, _sm(64))
    vals = oracle.fp16_value(v16).astype(np.float64)
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], vals[h // 2, 0])


def test_equal_keys_give_the_running_mean_of_v():
    rng = np.random.default_rng(9)
    n_kv, hd, P, T = 1, 64, 50, 10
    k16 = np.tile(oracle.fp16_bits(rng.standard_normal(hd).astype(np.float32)), (n_kv, P, 1))
    v16 = oracle.fp16_bits(rng.standard_normal((n_kv, P, hd)).astype(np.float32))
    q = rng.standard_normal((T, 2, hd)).astype(np.float32)
    out = oracle.chunk_attention(k16, v16, q, _sm(hd))
    vals = oracle.fp16_value(v16).astype(np.float64)[0]
    for t in range(T):
        np.testing.assert_allclose(out[t, 0], vals[: P - T + t + 1].mean(axis=0), rtol=1e-12, atol=1e-13)

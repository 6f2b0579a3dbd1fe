"""Pins for the oracle's paged store, float64 decode attention and compaction.

Attention is plain softmax attention over the dequantized cache (the split-K
partials and log-sum-exp combine of #3084 qwen35: FP16 K/V cache by default,
int8 with --kv-q8, "Extra Notes", only re-associate it).  It is pinned by
closed forms (one visible cell gives V, equal keys give the mean of V, two
cells give the logistic weights), by torch's scaled_dot_product_attention in
float64 (GQA by repeat_interleave, the verify window as an explicit mask),
and by properties (a shuffled block table gives bitwise the same result as
the identity table).  The stored cache is pinned against numpy's float16
conversion and the dequantized codes.
"""
import numpy as np
import pytest
import torch

import oracle

F16, Q8 = oracle.FMT_F16, oracle.FMT_Q8


def _identity_table(lens, bs):
    nbs = [max(1, -(-L // bs)) for L in lens]
    table = np.full((len(lens), max(nbs)), -1, np.int32)
    at = 0
    for b, nb in enumerate(nbs):
        table[b, :nb] = np.arange(at, at + nb)
        at += nb
    return table, sum(nbs)


def _fill(fmt, lens, n_kv, hd, bs, table, n_blocks, k, v):
    pool = oracle.PoolImage(fmt, n_kv, hd, bs, n_blocks)
    seq = np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    oracle.append(pool, k, v, seq, pos, table)
    return pool


def _logical(pool, table, lens):
    """Dequantized K/V per sequence [n_kv][L][hd] float64, read through numpy
    (float16 decode, code * scale) from the identity-table pool image."""
    out = []
    bs = pool.block_size
    for b, L in enumerate(lens):
        blocks = table[b, : max(1, -(-L // bs))]
        kk = pool.k[blocks]                    # [nb][n_kv][bs][hd]
        vv = pool.v[blocks]
        if pool.fmt == F16:
            kf = kk.view(np.float16).astype(np.float64)
            vf = vv.view(np.float16).astype(np.float64)
        else:
            ks = pool.ks[blocks].view(np.float16).astype(np.float64)
            vs = pool.vs[blocks].view(np.float16).astype(np.float64)
            kf = kk.astype(np.float64) * np.repeat(ks, 64, axis=-1)
            vf = vv.astype(np.float64) * np.repeat(vs, 64, axis=-1)
        kf = kf.transpose(1, 0, 2, 3).reshape(pool.n_kv, -1, pool.head_dim)[:, :L]
        vf = vf.transpose(1, 0, 2, 3).reshape(pool.n_kv, -1, pool.head_dim)[:, :L]
        out.append((kf, vf))
    return out


def _random_case(fmt, lens, n_kv, hd, bs, seed):
    rng = np.random.default_rng(seed)
    n = int(sum(lens))
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    k[rng.random((n, n_kv)) < 0.05] *= 10.0     # some large rows
    table, nb = _identity_table(lens, bs)
    return k, v, table, nb, _fill(fmt, lens, n_kv, hd, bs, table, nb, k, v)


@pytest.mark.parametrize("fmt", [F16, Q8])
def test_fp16_store_and_q8_roundtrip(fmt):
    lens, n_kv, hd, bs = [37, 5, 64], 3, 128, 16
    k, v, table, nb, pool = _random_case(fmt, lens, n_kv, hd, bs, 1)
    at = 0
    for (kf, vf), L in zip(_logical(pool, table, lens), lens):
        kx = k[at:at + L].transpose(1, 0, 2).astype(np.float64)
        vx = v[at:at + L].transpose(1, 0, 2).astype(np.float64)
        at += L
        if fmt == F16:   # the FP16 cache holds fp16(x), numpy's rounding
            assert np.array_equal(kf, kx.astype(np.float16).astype(np.float64))
            assert np.array_equal(vf, vx.astype(np.float16).astype(np.float64))
        else:            # int8: within half a scale step of x, group by group
            for xf, xx in ((kf, kx), (vf, vx)):
                s = np.abs(xx).reshape(n_kv, L, hd // 64, 64).max(-1) / 127.0
                bound = np.repeat(s, 64, axis=-1) * (0.5 + 2.0 ** -10)
                assert (np.abs(xf - xx) <= bound).all()


def test_shuffled_block_table_moves_whole_blocks():
    lens, n_kv, hd, bs = [70, 33], 2, 64, 16
    rng = np.random.default_rng(3)
    n = sum(lens)
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    table, nb = _identity_table(lens, bs)
    perm = rng.permutation(nb).astype(np.int32)
    shuffled = np.where(table >= 0, perm[np.maximum(table, 0)], -1).astype(np.int32)
    for fmt in (F16, Q8):
        a = _fill(fmt, lens, n_kv, hd, bs, table, nb, k, v)
        b = _fill(fmt, lens, n_kv, hd, bs, shuffled, nb, k, v)
        assert np.array_equal(b.k[perm], a.k) and np.array_equal(b.v[perm], a.v)
        if fmt == Q8:
            assert np.array_equal(b.ks[perm], a.ks) and np.array_equal(b.vs[perm], a.vs)
        q = rng.standard_normal((2, 2, 4, hd)).astype(np.float32)
        ctx = np.array(lens, np.int32)
        oa = oracle.attention(a, q, ctx, table, 0.125)
        ob = oracle.attention(b, q, ctx, shuffled, 0.125)
        assert np.array_equal(oa, ob)


@pytest.mark.parametrize("fmt", [F16, Q8])
def test_one_visible_cell_returns_its_value(fmt):
    n_kv, hd, bs, G = 2, 128, 16, 3
    k, v, table, nb, pool = _random_case(fmt, [1], n_kv, hd, bs, 4)
    q = np.random.default_rng(5).standard_normal((1, 1, n_kv * G, hd)).astype(np.float32)
    out = oracle.attention(pool, q, np.array([1], np.int32), table, 0.3)
    (kf, vf), = _logical(pool, table, [1])
    for h in range(n_kv * G):
        assert np.array_equal(out[0, 0, h], vf[h // G, 0])


@pytest.mark.parametrize("fmt", [F16, Q8])
def test_equal_keys_give_mean_of_values(fmt):
    n_kv, hd, bs, L = 1, 64, 16, 45
    rng = np.random.default_rng(6)
    k = np.repeat(rng.standard_normal((1, n_kv, hd)).astype(np.float32), L, axis=0)
    v = rng.standard_normal((L, n_kv, hd)).astype(np.float32)
    table, nb = _identity_table([L], bs)
    pool = _fill(fmt, [L], n_kv, hd, bs, table, nb, k, v)
    q = rng.standard_normal((1, 1, 4, hd)).astype(np.float32) * 3
    out = oracle.attention(pool, q, np.array([L], np.int32), table, 0.5)
    (kf, vf), = _logical(pool, table, [L])
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(vf[0].mean(0), (4, hd)),
                               rtol=0, atol=1e-13)


def test_two_cells_closed_form():
    # F16 cache with keys and query on one axis: z_i = sm * q0 * k_i exactly,
    # weights are the logistic function of z_0 - z_1.
    hd, bs = 64, 16
    k = np.zeros((2, 1, hd), np.float32)
    k[0, 0, 0], k[1, 0, 0] = 1.5, -0.75
    v = np.random.default_rng(8).standard_normal((2, 1, hd)).astype(np.float32)
    table, nb = _identity_table([2], bs)
    pool = _fill(F16, [2], 1, hd, bs, table, nb, k, v)
    q = np.zeros((1, 1, 1, hd), np.float32)
    q[0, 0, 0, 0] = 2.0
    sm = 0.25
    out = oracle.attention(pool, q, np.array([2], np.int32), table, sm)
    z0, z1 = sm * 2.0 * 1.5, sm * 2.0 * -0.75
    w0 = 1.0 / (1.0 + np.exp(z1 - z0))
    v16 = v.astype(np.float16).astype(np.float64)
    np.testing.assert_allclose(out[0, 0, 0], w0 * v16[0, 0] + (1 - w0) * v16[1, 0],
                               rtol=0, atol=1e-14)


def _sdpa(kf, vf, q, L, W, G, sm):
    """torch scaled_dot_product_attention (float64) for one sequence."""
    n_kv = kf.shape[0]
    K = torch.from_numpy(kf).repeat_interleave(G, dim=0)[None]     # [1][n_q][L][hd]
    V = torch.from_numpy(vf).repeat_interleave(G, dim=0)[None]
    Q = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]  # [1][n_q][W][hd]
    # verify window: query w is cell L - W + w and sees cells up to itself
    mask = torch.arange(L)[None, :] <= (L - W + torch.arange(W))[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(
        Q, K, V, attn_mask=mask, scale=float(np.float64(np.float32(sm))))
    return out[0].permute(1, 0, 2).numpy()                          # [W][n_q][hd]


@pytest.mark.parametrize("fmt,n_kv,G,hd,W", [
    (F16, 1, 4, 128, 1), (Q8, 1, 4, 128, 1), (F16, 4, 2, 64, 3),
    (Q8, 3, 4, 128, 4), (Q8, 2, 8, 256, 1), (F16, 2, 1, 256, 2),
])
def test_matches_torch_sdpa(fmt, n_kv, G, hd, W):
    lens, bs = [300, 17, 129], 32
    k, v, table, nb, pool = _random_case(fmt, lens, n_kv, hd, bs, 11 + hd + W)
    rng = np.random.default_rng(12)
    q = rng.standard_normal((len(lens), W, n_kv * G, hd)).astype(np.float32)
    sm = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    out = oracle.attention(pool, q, np.array(lens, np.int32), table, sm)
    for b, (kf, vf) in enumerate(_logical(pool, table, lens)):
        ref = _sdpa(kf, vf, q[b], lens[b], W, G, sm)
        np.testing.assert_allclose(out[b], ref, rtol=1e-10, atol=1e-10)


def test_queries_without_visible_cells_are_zero():
    n_kv, hd, bs = 1, 64, 16
    k, v, table, nb, pool = _random_case(F16, [3, 2], n_kv, hd, bs, 13)
    q = np.ones((3, 4, 2, hd), np.float32)
    table3 = np.vstack([table, table[:1]])
    out = oracle.attention(pool, q, np.array([3, 2, 0], np.int32), table3, 0.1)
    assert np.isfinite(out).all()
    assert not out[0, 0].any()               # L=3, W=4: token 0 sees nothing
    assert out[0, 1:].any()
    assert not out[1, :2].any() and out[1, 2:].any()
    assert not out[2].any()                  # empty sequence


@pytest.mark.parametrize("fmt", [F16, Q8])
def test_compaction(fmt):
    lens, n_kv, hd, bs = [75], 2, 128, 16
    k, v, table, nb, pool = _random_case(fmt, lens, n_kv, hd, bs, 14)
    rng = np.random.default_rng(15)
    perm = rng.permutation(nb).astype(np.int32)
    shuffled = perm[table]
    pool_s = _fill(fmt, lens, n_kv, hd, bs, shuffled, nb, k, v)
    ok, ov = oracle.compact_f16(pool_s, shuffled[0], lens[0])
    (kf, vf), = _logical(pool, table, lens)
    # the dequantized values are exact products; their fp16 rounding (numpy)
    assert np.array_equal(ok, kf.astype(np.float16).view(np.uint16))
    assert np.array_equal(ov, vf.astype(np.float16).view(np.uint16))
    if fmt == F16:   # a pure copy of the stored bits
        assert np.array_equal(ok.view(np.float16).astype(np.float32),
                              k.transpose(1, 0, 2).astype(np.float16).astype(np.float32))


def test_parallel_build_is_bitwise_the_single_threaded_oracle():
    """The OpenMP build (the multi-core CPU baseline) runs the same rows with
    the same arithmetic, so its output equals the plain build's bit for bit."""
    path = oracle.parallel_library(4)
    if path is None:
        pytest.skip("gcc without OpenMP")
    lens, n_kv, hd, bs, G, W = [301, 77, 512], 2, 128, 32, 4, 3
    for fmt in (F16, Q8):
        k, v, table, nb, pool = _random_case(fmt, lens, n_kv, hd, bs, 7)
        q = np.random.default_rng(8).standard_normal((len(lens), W, n_kv * G, hd)).astype(np.float32)
        ctx = np.array(lens, np.int32)
        ref = oracle.attention(pool, q, ctx, table, 0.0883883)
        with oracle.use_library(path) as u:
            assert u._lib.kvo_threads() == 4
            par = oracle.attention(pool, q, ctx, table, 0.0883883)
        assert np.array_equal(ref.view(np.uint64), par.view(np.uint64))

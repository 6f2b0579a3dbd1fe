"""Pins for the oracle's K8V4 format: int8 K and rotated Q4_0 V.

#711 kv: --kv k8v4 streams with --kv-resident, "What": INT8 K with rotated
Q4_0 V at 816 B per cell (the byte count is pinned in test_oracle_sizing).
The page names the rotation and the 4-bit format but neither's details; the
oracle reads them as the Walsh-Hadamard transform (Sylvester order, entries
+-1, no normalisation; its inverse is itself divided by the row length) and
Q4_0 over 32 rotated dims: d = fp16(m / -8) for m the block's element of
largest magnitude (the first on ties), code = clamp(rint(y / d), -8, 7) + 8,
value (code - 8) * d, two codes a byte (dim 2j low nibble, 2j + 1 high).

Pinned by scipy's Hadamard matrix (the transform and its order), by rows
designed in the rotated basis (y chosen, x = H y / n, so that the fp32
transform is exact and every code and scale is known in advance: ties of
magnitude and of rounding, nibble order, a zero block), by the error bound
of 4-bit codes on random rows, by attention against torch's
scaled_dot_product_attention over K and V decoded here with numpy and
scipy, and by compaction against the same decoding.
"""
import numpy as np
import pytest
import torch
from scipy.linalg import hadamard

import oracle

K8V4 = oracle.FMT_K8V4


def _unpack(codes):
    """uint8 [..., hd/2] -> ints [..., hd]: dim 2j low nibble, 2j + 1 high."""
    lo = (codes & 15).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,))


def _decode_rotated(codes, scales):
    d = scales.view(np.float16).astype(np.float64)
    return (_unpack(codes) - 8) * np.repeat(d, 32, axis=-1)


def _from_rotated(y):
    """x with H x = y exactly in fp32 (y small integers, n a power of two)."""
    n = y.shape[-1]
    return (y.astype(np.float64) @ hadamard(n).T / n).astype(np.float32)


@pytest.mark.parametrize("n", [2, 32, 64, 128, 256])
def test_transform_is_sylvester_hadamard(n):
    rng = np.random.default_rng(n)
    x = rng.integers(-50, 50, (3, n)).astype(np.float32)   # exact in fp32
    y = oracle.hadamard_f32(x)
    np.testing.assert_array_equal(y.astype(np.float64), x.astype(np.float64) @ hadamard(n).T)
    np.testing.assert_array_equal(oracle.hadamard_f32(y), n * x)   # H H = n I
    xr = rng.standard_normal((4, n)).astype(np.float32)
    np.testing.assert_allclose(oracle.hadamard_f32(xr), xr.astype(np.float64) @ hadamard(n).T,
                               rtol=0, atol=1e-5 * np.sqrt(n))


def test_designed_block_scale_codes_and_nibble_order():
    hd = 64
    y = np.zeros(hd)
    # block 0: maximum +5 at dim 3 and -5 at dim 10: the first wins, d = -0.625
    y[3], y[10], y[4], y[5] = 5, -5, 1.25, -2.5
    # block 1: maximum 8 at dim 33: d = -1; y / d = -2.5 and -1.5 are ties
    y[33], y[34], y[35], y[36], y[37] = 8, 2.5, 1.5, 0.5, -7
    x = _from_rotated(y[None])
    assert np.array_equal(oracle.hadamard_f32(x).astype(np.float64), y[None])
    codes, scales = oracle.quantize_rows_q4r(x)
    d = scales.view(np.float16).astype(np.float64)[0]
    assert d[0] == -0.625 and d[1] == -1.0
    c = _unpack(codes)[0]
    assert c[3] == 0 and c[10] == 15              # -8 and clamp(+8) = 7
    assert c[4] == 6 and c[5] == 12               # -2, +4
    assert c[33] == 0 and c[37] == 15             # -8, +7
    assert c[34] == 6 and c[35] == 6 and c[36] == 8   # rint: -2.5 -> -2, -1.5 -> -2, -0.5 -> 0
    assert (c[[i for i in range(hd) if y[i] == 0]] == 8).all()
    # byte j holds dims 2j (low) and 2j + 1 (high)
    assert codes[0, 1] == c[2] | (c[3] << 4) and codes[0, 2] == c[4] | (c[5] << 4)


def test_zero_block_gives_zero_scale_and_offset_codes():
    hd = 128
    y = np.zeros(hd)
    y[40:64] = np.arange(1, 25)                   # block 1 only
    codes, scales = oracle.quantize_rows_q4r(_from_rotated(y[None]))
    d = scales.view(np.float16).astype(np.float64)[0]
    assert d[0] == 0 and d[2] == 0 and d[3] == 0 and d[1] == -3.0
    c = _unpack(codes)[0]
    assert (c[:32] == 8).all() and (c[64:] == 8).all()


def test_random_rows_within_half_a_step():
    rng = np.random.default_rng(31)
    for hd in (64, 128, 256):
        x = rng.standard_normal((200, hd)).astype(np.float32)
        x[::7] *= 20.0
        codes, scales = oracle.quantize_rows_q4r(x)
        y = x.astype(np.float64) @ hadamard(hd).T
        deq = _decode_rotated(codes, scales)
        d = np.repeat(np.abs(scales.view(np.float16).astype(np.float64)), 32, axis=-1)
        ratio = y / np.where(d == 0, 1, d)
        inside = np.abs(ratio) <= 7.5             # not clamped at the +7 end
        slack = 1e-5 * np.abs(y).max(-1, keepdims=True)   # the fp32 transform
        assert (np.abs(deq - y) <= d / 2 * (1 + 2**-9) + slack)[inside].all()
        # the block maximum is code 0 (value -8 d, m up to d's fp16 rounding)
        yb = y.reshape(len(x), hd // 32, 32)
        first = np.abs(yb).argmax(-1)
        cb = _unpack(codes).reshape(len(x), hd // 32, 32)
        assert (np.take_along_axis(cb, first[..., None], -1) == 0).all()
        db = scales.view(np.float16).astype(np.float64)
        m = np.take_along_axis(yb, first[..., None], -1)[..., 0]
        np.testing.assert_allclose(-8 * db, m, rtol=2**-10, atol=1e-4)


def _case(lens, n_kv, hd, bs, seed):
    rng = np.random.default_rng(seed)
    n = int(sum(lens))
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v[rng.random((n, n_kv)) < 0.05] *= 10.0
    nbs = [max(1, -(-L // bs)) for L in lens]
    table = np.full((len(lens), max(nbs)), -1, np.int32)
    perm = rng.permutation(sum(nbs)).astype(np.int32)
    at = 0
    for b, nb in enumerate(nbs):
        table[b, :nb] = perm[at:at + nb]
        at += nb
    pool = oracle.PoolImage(K8V4, n_kv, hd, bs, sum(nbs))
    seq = np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    oracle.append(pool, k, v, seq, pos, table)
    return k, v, table, pool


def _logical(pool, table, b, L):
    """Decoded K and V [n_kv][L][hd] float64 of sequence b: K = code * scale,
    V = H (decoded rotated row) / hd, read here with numpy and scipy."""
    hd = pool.head_dim
    blocks = table[b, : max(1, -(-L // pool.block_size))]
    ks = pool.ks[blocks].view(np.float16).astype(np.float64)
    kf = pool.k[blocks].astype(np.float64) * np.repeat(ks, 64, axis=-1)
    vr = _decode_rotated(pool.v[blocks], pool.vs[blocks])
    vf = vr @ hadamard(hd).T / hd
    fix = lambda a: a.transpose(1, 0, 2, 3).reshape(pool.n_kv, -1, hd)[:, :L]
    return fix(kf), fix(vf)


def test_stored_codes_are_the_row_quantizers():
    lens, n_kv, hd, bs = [37, 20], 2, 128, 16
    k, v, table, pool = _case(lens, n_kv, hd, bs, 32)
    ck, sk = oracle.quantize_rows_q8(k)
    cv, sv = oracle.quantize_rows_q4r(v)
    at = 0
    for b, L in enumerate(lens):
        for p in range(L):
            blk, slot = table[b, p // bs], p % bs
            for h in range(n_kv):
                assert np.array_equal(pool.k[blk, h, slot], ck[at + p, h])
                assert np.array_equal(pool.ks[blk, h, slot], sk[at + p, h])
                assert np.array_equal(pool.v[blk, h, slot], cv[at + p, h])
                assert np.array_equal(pool.vs[blk, h, slot], sv[at + p, h])
        at += L


def test_one_visible_cell_returns_its_derotated_value():
    n_kv, hd, bs, G = 2, 256, 16, 4
    k, v, table, pool = _case([1], n_kv, hd, bs, 33)
    q = np.random.default_rng(34).standard_normal((1, 1, n_kv * G, hd)).astype(np.float32)
    out = oracle.attention(pool, q, np.array([1], np.int32), table, 0.2)
    _, vf = _logical(pool, table, 0, 1)
    for h in range(n_kv * G):
        np.testing.assert_allclose(out[0, 0, h], vf[h // G, 0], rtol=0, atol=1e-12)
    # and the rotated 4-bit V is close to the appended row
    np.testing.assert_allclose(vf[:, 0], v[0].astype(np.float64), rtol=0,
                               atol=0.1 * np.abs(v).max())


@pytest.mark.parametrize("n_kv,G,hd,W", [(1, 4, 128, 1), (2, 4, 256, 3), (2, 2, 64, 2)])
def test_matches_torch_sdpa(n_kv, G, hd, W):
    lens, bs = [150, 33, 64], 16
    k, v, table, pool = _case(lens, n_kv, hd, bs, 35 + hd + W)
    q = np.random.default_rng(36).standard_normal((len(lens), W, n_kv * G, hd)).astype(np.float32)
    sm = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    out = oracle.attention(pool, q, np.array(lens, np.int32), table, sm)
    for b, L in enumerate(lens):
        kf, vf = _logical(pool, table, b, L)
        K = torch.from_numpy(kf).repeat_interleave(G, dim=0)[None]
        V = torch.from_numpy(vf).repeat_interleave(G, dim=0)[None]
        Q = torch.from_numpy(q[b].astype(np.float64)).permute(1, 0, 2)[None]
        mask = torch.arange(L)[None, :] <= (L - W + torch.arange(W))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, attn_mask=mask, scale=float(np.float64(np.float32(sm))))
        np.testing.assert_allclose(out[b], ref[0].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-10)


def test_compaction_derotates_v():
    lens, n_kv, hd, bs = [70], 2, 128, 16
    k, v, table, pool = _case(lens, n_kv, hd, bs, 37)
    ok, ov = oracle.compact_f16(pool, table[0], lens[0])
    kf, vf = _logical(pool, table, 0, lens[0])
    assert np.array_equal(ok, kf.astype(np.float16).view(np.uint16))   # exact products
    # V: the fp32 transform may round where float64 does not: within one fp16 step
    got = ov.view(np.float16).astype(np.float64)
    want = vf.astype(np.float16).astype(np.float64)
    step = np.spacing(np.abs(want).astype(np.float16)).astype(np.float64)
    assert (np.abs(got - want) <= step).all()
    assert np.mean(got == want) > 0.95


def test_compaction_exact_when_every_block_shares_its_scale():
    # rows designed in the rotated basis with one scale for every block: the
    # fp32 transform of the decoded row is exact, so compaction is
    # fp16(H y / n) of float64, bit for bit
    hd, bs, n = 64, 16, 16
    rng = np.random.default_rng(38)
    y = rng.integers(-7, 8, (n, 1, hd)).astype(np.float64)
    y[:, :, ::32] = 8                              # every block: maximum 8, d = -1
    x = _from_rotated(y.reshape(n, hd)).reshape(n, 1, hd)
    pool = oracle.PoolImage(K8V4, 1, hd, bs, 1)
    oracle.append(pool, x, x, np.zeros(n, np.int32), np.arange(n, dtype=np.int32),
                  np.zeros((1, 1), np.int32))
    _, ov = oracle.compact_f16(pool, np.zeros(1, np.int32), n)
    dec = _decode_rotated(pool.v[0, 0], pool.vs[0, 0])
    assert np.array_equal(dec, np.clip(np.rint(-y[:, 0]), -8, 7) * -1.0)
    want = (dec @ hadamard(hd).T / hd).astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ov[0], want)


def test_geometry_needs_a_power_of_two_multiple_of_64():
    with pytest.raises(RuntimeError):
        pool = oracle.PoolImage(K8V4, 1, 192, 16, 1)
        x = np.zeros((1, 1, 192), np.float32)
        oracle.append(pool, x, x, np.zeros(1, np.int32), np.zeros(1, np.int32),
                      np.zeros((1, 1), np.int32))

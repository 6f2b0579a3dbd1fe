"""Pins for the oracle's gather / scatter of a sequence's cells.

What is saved for a sequence is its used cells' K/V bytes followed by their
scales, token-major (Path F format v3: persist per-head INT8 KV scales for
INT8 + persistent KV interop, "Scope"), and int8 codes never travel without
their scales (same page, "Why": int8 bytes without the scales hydrate to
garbage).  Pinned by the stored values themselves (numpy float16 of the
input for FP16; the row quantizer for int8, pinned in test_oracle_quant),
by scatter into a pool with another block table followed by gather (the
identity), by attention being unchanged after the move, and by the refusal
of int8 without scales.
"""
import numpy as np
import pytest

import oracle

F16, Q8, K8V4 = oracle.FMT_F16, oracle.FMT_Q8, oracle.FMT_K8V4


def _pool(fmt, n_kv, hd, bs, nb, table_row, k, v):
    pool = oracle.PoolImage(fmt, n_kv, hd, bs, nb)
    n = k.shape[0]
    oracle.append(pool, k, v, np.zeros(n, np.int32), np.arange(n, dtype=np.int32), table_row[None])
    return pool


@pytest.mark.parametrize("fmt", [F16, Q8, K8V4])
def test_gather_returns_the_stored_rows_in_order(fmt):
    rng = np.random.default_rng(21)
    n, n_kv, hd, bs = 45, 2, 128, 16
    nb = -(-n // bs)
    row = rng.permutation(nb).astype(np.int32)
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    pool = _pool(fmt, n_kv, hd, bs, nb, row, k, v)
    ck, cv, sk, sv = oracle.gather_cells(pool, row, n)
    if fmt == F16:
        np.testing.assert_array_equal(ck, k.astype(np.float16).view(np.uint16))
        np.testing.assert_array_equal(cv, v.astype(np.float16).view(np.uint16))
        assert sk is None and sv is None
    else:
        v_rows = oracle.quantize_rows_q8 if fmt == Q8 else oracle.quantize_rows_q4r
        for x, c, s, rows in ((k, ck, sk, oracle.quantize_rows_q8), (v, cv, sv, v_rows)):
            codes, scales = rows(x.reshape(-1, hd))
            np.testing.assert_array_equal(c.reshape(codes.shape), codes)
            np.testing.assert_array_equal(s.reshape(scales.shape), scales)
            assert c.shape[:2] == s.shape[:2] == (n, n_kv)


@pytest.mark.parametrize("fmt", [F16, Q8, K8V4])
def test_scatter_into_another_layout_then_gather_is_the_identity(fmt):
    rng = np.random.default_rng(22)
    n, n_kv, hd, bs = 70, 3, 64, 32
    nb = -(-n // bs)
    row_a = np.arange(nb, dtype=np.int32)
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    a = _pool(fmt, n_kv, hd, bs, nb, row_a, k, v)
    saved = oracle.gather_cells(a, row_a, n)
    # a pool with more blocks and the cells in other blocks
    b = oracle.PoolImage(fmt, n_kv, hd, bs, nb + 3)
    row_b = rng.permutation(nb + 3)[:nb].astype(np.int32)
    oracle.scatter_cells(b, row_b, *saved)
    back = oracle.gather_cells(b, row_b, n)
    for x, y in zip(saved, back):
        if x is None:
            assert y is None
        else:
            np.testing.assert_array_equal(x, y)
    # attention over the moved cells is unchanged, bit for bit
    q = rng.standard_normal((1, 2, 2 * n_kv, hd)).astype(np.float32)
    ctx = np.array([n], np.int32)
    oa = oracle.attention(a, q, ctx, row_a[None], 0.125)
    ob = oracle.attention(b, q, ctx, row_b[None], 0.125)
    np.testing.assert_array_equal(oa, ob)


def test_int8_codes_without_scales_are_refused():
    rng = np.random.default_rng(23)
    n, n_kv, hd, bs = 16, 1, 64, 16
    row = np.zeros(1, np.int32)
    x = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    pool = _pool(Q8, n_kv, hd, bs, 1, row, x, x)
    ck, cv, sk, sv = oracle.gather_cells(pool, row, n)
    with pytest.raises(RuntimeError):
        oracle.scatter_cells(pool, row, ck, cv, None, None)

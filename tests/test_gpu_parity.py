"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

The five workloads run at their full sizes, in the launch configuration the
benchmark uses (the library plans splits itself), with every output compared:
cache codes / scales / fp16 values and compaction bit-exact, attention within
max-abs 2e-3 and relative L2 1e-3.  Reduced-size copies cover shape and
edge cases (head dims, block sizes, GQA groups, verify windows, ragged and
empty contexts, degenerate quantization groups) and the bitwise invariants
(paged equals contiguous, one-at-a-time append equals one chunk).
"""
import numpy as np
import pytest
import torch

import workloads
import quantized_kv_cache_append_gb300 as kvq
from tests.gpu_pairs import Pair, assert_attention_close, dev, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.fail("the GPU suite needs a CUDA device")
    kvq.build()
    kvq.load_library()


def _prefilled(wl, fmt):
    p = Pair(fmt, wl.n_kv, wl.head_dim, wl.block_size, wl.n_blocks, wl.block_table)
    p.append(wl.k, wl.v, wl.tok_seq, wl.tok_pos)
    return p


# --------------------------------------------------------------------------
# the five workloads at full size
# --------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["f16", "q8", "k8v4"])
def test_tiny(fmt):
    wl = workloads.make("tiny")
    p = _prefilled(wl, fmt)
    p.assert_cache_equal()
    p.check_decode(wl.q, wl.ctx_lens, wl.sm_scale)
    p.check_compact(0, int(wl.ctx_lens[0]))


@pytest.mark.parametrize("fmt", ["f16", "q8", "k8v4"])
def test_gqa32k_append_decode_steps(fmt):
    wl = workloads.make("gqa32k")
    p = _prefilled(wl, fmt)
    p.check_decode(wl.q, wl.ctx_lens, wl.sm_scale)
    checked = {0, 1, 2, 31, 63}
    for i, st in enumerate(wl.steps):
        p.append(st["k"], st["v"], st["tok_seq"], st["tok_pos"])
        if i in checked:
            p.check_decode(st["q"], st["ctx_lens"], wl.sm_scale)
    p.assert_cache_equal()


@pytest.mark.parametrize("fmt", ["q8", "k8v4"])
def test_ragged_paged_batch(fmt):
    wl = workloads.make("ragged")
    p = _prefilled(wl, fmt)
    p.assert_cache_equal()
    p.check_decode(wl.q, wl.ctx_lens, wl.sm_scale)


@pytest.mark.parametrize("fmt", ["f16", "q8", "k8v4"])
def test_long256k(fmt):
    wl = workloads.make("long256k")
    p = _prefilled(wl, fmt)
    p.assert_cache_equal()
    p.check_decode(wl.q, wl.ctx_lens, wl.sm_scale)


@pytest.mark.parametrize("fmt", ["q8", "k8v4"])
def test_chunk_compact_verify(fmt):
    wl = workloads.make("chunk_verify")
    p = _prefilled(wl, fmt)
    c = wl.chunk
    p.append(c["k"], c["v"], c["tok_seq"], c["tok_pos"])
    p.assert_cache_equal()
    L = int(c["ctx_lens"][0])
    p.check_compact(0, L)
    p.check_decode(wl.q, c["ctx_lens"], wl.sm_scale)


# --------------------------------------------------------------------------
# shapes and edge cases at reduced size
# --------------------------------------------------------------------------

def _random_pair(fmt, lens, n_kv, hd, bs, seed, shuffle=True):
    rng = np.random.default_rng(seed)
    nbs = [max(1, -(-L // bs)) for L in lens]
    nb = sum(nbs)
    perm_rng = np.random.default_rng(seed + 7919)          # data draws do not depend on it
    perm = perm_rng.permutation(nb).astype(np.int32) if shuffle else np.arange(nb, dtype=np.int32)
    table = np.full((len(lens), max(nbs)), -1, np.int32)
    at = 0
    for b, n in enumerate(nbs):
        table[b, :n] = perm[at:at + n]
        at += n
    n = int(sum(lens))
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    big = rng.random((n, n_kv)) < 0.02
    k[big] *= 10.0
    v[big] *= 10.0
    seq = np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    p = Pair(fmt, n_kv, hd, bs, nb, table)
    if n:
        p.append(k, v, seq, pos)
    return p, rng


@pytest.mark.parametrize("fmt", ["f16", "q8", "k8v4"])
@pytest.mark.parametrize("hd,bs,n_kv,G,W", [
    (64, 16, 2, 1, 1), (64, 64, 1, 2, 16), (128, 256, 3, 4, 2), (128, 32, 2, 1, 4),
    (128, 1024, 1, 8, 2), (256, 128, 2, 8, 1), (256, 16, 1, 2, 4), (64, 512, 4, 8, 4),
])
def test_shapes(fmt, hd, bs, n_kv, G, W):
    lens = [W, 1 + W, 37, 300, 2049]
    p, rng = _random_pair(fmt, lens, n_kv, hd, bs, seed=hd * 7 + bs + G * 3 + W)
    p.assert_cache_equal()
    q = rng.standard_normal((len(lens), W, n_kv * G, hd)).astype(np.float32)
    sm = workloads.sm_scale_for(hd)
    p.check_decode(q, lens, sm)
    p.check_decode(q, lens, sm, max_ctx=p.bt_host.shape[1] * bs)   # widest allowed plan
    p.check_compact(4, lens[4])


@pytest.mark.parametrize("fmt", ["f16", "q8", "k8v4"])
@pytest.mark.parametrize("hd,n_kv,G,W", [
    (256, 2, 8, 2), (256, 2, 8, 4), (256, 1, 4, 4), (256, 1, 2, 16),   # 16, 32, 16, 32 rows
    (128, 2, 8, 4), (128, 1, 4, 8), (128, 3, 2, 16), (128, 1, 8, 3),   # 32, 32, 32, 24 rows
    (64, 2, 8, 4), (64, 1, 4, 8),                                      # 32 rows in one CTA
])
def test_wide_verify_windows(fmt, hd, n_kv, G, W):
    """Verify windows whose G * W query rows exceed one CTA's row tile (8
    rows at head_dim 256, 16 at 128) are cut into row tiles; every tile
    must give the oracle's attention, causal limits included (#711 kv:
    --kv k8v4 streams with --kv-resident, "How": verify-window appends;
    "Measured": spec 4)."""
    lens = [W, 2 * W + 5, 700, 3001]
    p, rng = _random_pair(fmt, lens, n_kv, hd, 64, seed=hd + 11 * G + W + n_kv)
    q = rng.standard_normal((len(lens), W, n_kv * G, hd)).astype(np.float32)
    sm = workloads.sm_scale_for(hd)
    p.check_decode(q, lens, sm)
    p.check_decode(q, lens, sm, max_ctx=p.bt_host.shape[1] * 64)   # widest allowed plan


@pytest.mark.parametrize("fmt", ["f16", "q8", "k8v4"])
def test_single_cell_outputs_its_value(fmt):
    p, rng = _random_pair(fmt, [1], 2, 128, 16, seed=3)
    q = rng.standard_normal((1, 1, 8, 128)).astype(np.float32)
    got = p.decode_gpu(q, np.array([1], np.int32), 1, 0.1)
    ref = p.decode_oracle(q, np.array([1], np.int32), 0.1)
    if fmt == "k8v4":   # the fp32 inverse rotation rounds: within the bar
        assert_attention_close(got, ref)
    else:
        assert np.array_equal(got.astype(np.float64), ref)   # exp(0) / 1 * v: exact


def test_empty_sequences_give_zero_output():
    p, rng = _random_pair("q8", [0, 5, 0, 300], 2, 128, 16, seed=4)
    q = rng.standard_normal((4, 1, 4, 128)).astype(np.float32)
    got, ref = p.check_decode(q, [0, 5, 0, 300], 0.09)
    assert not got[0].any() and not got[2].any()


@pytest.mark.parametrize("reps", [1, 24])   # a few tokens, and the bulk kernel shape
def test_degenerate_quantization_groups(reps):
    # zero rows, tiny rows (fp16-subnormal or underflowing scales), huge rows
    # (scale overflows to +inf: zero codes), exact ties, fp32 subnormal inputs
    rng = np.random.default_rng(5)
    n, n_kv, hd = 64, 2, 256
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    k[0] = 0.0
    k[1] *= 1e-7
    k[2] *= 3e-4
    k[3] *= 2e6
    k[4, :, :] = np.float32(127.0)
    k[4, :, 1::2] = np.float32(2.5)
    k[5] = np.float32(1e-40)                   # fp32 subnormals
    k[6, 0, :64] = np.float32(260223.0 / 2048.0)
    k[6, 0, 1] = np.float32(65.51)
    v = k[::-1].copy()
    k, v = np.tile(k, (reps, 1, 1)), np.tile(v, (reps, 1, 1))
    n *= reps
    table = np.arange(-(-n // 16), dtype=np.int32)[None]
    for fmt in ("f16", "q8", "k8v4"):
        p = Pair(fmt, n_kv, hd, 16, table.shape[1], table)
        p.append(k, v, np.zeros(n, np.int32), np.arange(n, dtype=np.int32))
        p.assert_cache_equal()


@pytest.mark.parametrize("reps", [1, 12])
def test_quantization_ties_and_near_ties(reps):
    # Groups whose maximum is exactly 127 s (s an fp16 value, so the stored
    # scale is s itself) and whose other elements are (k + 1/2) s exactly or
    # 1-3 fp32 ulps away: x / s is an exact half-integer (round half to even)
    # or so close to one that only the IEEE quotient decides.
    rng = np.random.default_rng(11)
    n, n_kv, hd = 96, 2, 128
    s = rng.uniform(2.0 ** -10, 16.0, size=(n, n_kv, hd // 64)).astype(np.float16)
    s = s.astype(np.float32)
    half = rng.integers(-127, 127, size=(n, n_kv, hd)).astype(np.float32) + np.float32(0.5)
    x = (half * np.repeat(s, 64, axis=-1)).astype(np.float32)
    steps = rng.integers(-3, 4, size=x.shape)
    for k in (1, 2, 3):
        up, dn = steps >= k, steps <= -k
        x[up] = np.nextafter(x[up], np.float32(np.inf))
        x[dn] = np.nextafter(x[dn], np.float32(-np.inf))
    x[..., ::64] = (np.float32(127.0) * s).astype(np.float32)   # the group maxima
    v = -x[::-1].copy()
    x, v = np.tile(x, (reps, 1, 1)), np.tile(v, (reps, 1, 1))
    n *= reps
    table = np.arange(-(-n // 16), dtype=np.int32)[None]
    p = Pair("q8", n_kv, hd, 16, table.shape[1], table)
    p.append(x, v, np.zeros(n, np.int32), np.arange(n, dtype=np.int32))
    p.assert_cache_equal()


@pytest.mark.parametrize("reps", [1, 16])
def test_scale_rounding_midpoints(reps):
    # Group maxima a with a / 127 on, or a few fp32 ulps from, a midpoint
    # between two fp16 values (where fp16(a / 127) is decided by the last
    # bits of the fp32 quotient), and maxima whose scale is an fp16
    # subnormal or near the fp16 maximum.
    rng = np.random.default_rng(12)
    n, n_kv, hd = 64, 2, 128
    x = rng.uniform(-1.0, 1.0, size=(n, n_kv, hd)).astype(np.float32)
    ng = n * n_kv * (hd // 64)
    h = rng.uniform(2.0 ** -13, 500.0, size=ng).astype(np.float16)
    h_next = np.nextafter(h, np.float16(np.inf))
    mid = (h.astype(np.float64) + h_next.astype(np.float64)) / 2.0
    a = (mid * 127.0).astype(np.float32)
    shift = rng.integers(-3, 4, size=ng)
    for k in (1, 2, 3):
        a[shift >= k] = np.nextafter(a[shift >= k], np.float32(np.inf))
        a[shift <= -k] = np.nextafter(a[shift <= -k], np.float32(-np.inf))
    a[:16] = rng.uniform(1e-7, 6e-3, size=16).astype(np.float32)        # fp16-subnormal scales
    a[16:24] = np.float32(65504.0 * 127.0) * rng.uniform(0.999, 1.001, size=8).astype(np.float32)
    groups = x.reshape(ng, 64)
    groups *= (a / np.abs(groups).max(axis=1))[:, None]
    groups[np.arange(ng), rng.integers(0, 64, size=ng)] = a * np.where(rng.random(ng) < 0.5, 1, -1)
    x = groups.reshape(n, n_kv, hd).astype(np.float32)
    v = x[::-1].copy()
    x, v = np.tile(x, (reps, 1, 1)), np.tile(v, (reps, 1, 1))
    n *= reps
    table = np.arange(-(-n // 16), dtype=np.int32)[None]
    p = Pair("q8", n_kv, hd, 16, table.shape[1], table)
    p.append(x, v, np.zeros(n, np.int32), np.arange(n, dtype=np.int32))
    p.assert_cache_equal()


def test_paged_equals_contiguous_bitwise():
    lens = [700, 1500]
    for fmt in ("f16", "q8", "k8v4"):
        outs = []
        for shuffle in (False, True):
            p, rng = _random_pair(fmt, lens, 2, 128, 64, seed=6, shuffle=shuffle)
            q = np.random.default_rng(9).standard_normal((2, 1, 8, 128)).astype(np.float32)
            max_ctx = p.bt_host.shape[1] * 64                   # table width in cells
            outs.append(p.decode_gpu(q, np.array(lens, np.int32), max_ctx, 0.088))
        assert np.array_equal(outs[0], outs[1])


def test_one_at_a_time_append_equals_chunk():
    n, n_kv, hd, bs = 300, 2, 128, 32
    rng = np.random.default_rng(10)
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    table = rng.permutation(10).astype(np.int32)[None]
    for fmt in ("f16", "q8", "k8v4"):
        a = Pair(fmt, n_kv, hd, bs, 10, table)
        b = Pair(fmt, n_kv, hd, bs, 10, table)
        a.append(k, v, np.zeros(n, np.int32), np.arange(n, dtype=np.int32))
        for i in range(0, n, 37):
            j = min(n, i + 37)
            b.gpu.append(dev(k[i:j]), dev(v[i:j]), dev(np.zeros(j - i, np.int32)),
                         dev(np.arange(i, j, dtype=np.int32)), b.bt)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(a.gpu.k), host_bits(b.gpu.k))
        assert np.array_equal(host_bits(a.gpu.v), host_bits(b.gpu.v))
        if fmt != "f16":
            assert np.array_equal(host_bits(a.gpu.ks), host_bits(b.gpu.ks))
            assert np.array_equal(host_bits(a.gpu.vs), host_bits(b.gpu.vs))


def test_out_of_range_block_ids_are_skipped_not_followed():
    # Broken preconditions must not turn into stray memory accesses: the
    # kernels check every block id against the pool and skip (append,
    # compaction) or zero (attention) the cells whose id is out of range.
    n_kv, hd, bs = 2, 128, 16
    table = np.array([[0, 1, -5, 1 << 28]], np.int32)
    rng = np.random.default_rng(11)
    for fmt in ("f16", "q8", "k8v4"):
        p = Pair(fmt, n_kv, hd, bs, 2, table)
        n = 64
        k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
        p.gpu.append(dev(k), dev(k), dev(np.zeros(n, np.int32)),
                     dev(np.arange(n, dtype=np.int32)), p.bt)
        q = rng.standard_normal((1, 1, 4, hd)).astype(np.float32)
        out = p.decode_gpu(q, np.array([n], np.int32), n, 0.1)
        zeros = torch.zeros((n_kv, n, hd), dtype=torch.float16, device="cuda")
        ok, ov = p.gpu.compact(dev(table[0]), n, out_k=zeros, out_v=zeros.clone())
        torch.cuda.synchronize()
        assert np.isfinite(out).all()
        assert not host_bits(ok)[:, 32:].any()      # cells of the bad blocks were skipped


def test_validation_with_real_buffers():
    p, rng = _random_pair("q8", [64], 2, 128, 16, seed=12)
    q = dev(rng.standard_normal((1, 1, 4, 128)).astype(np.float32))
    out = torch.empty_like(q)
    ctx = dev(np.array([64], np.int32))
    ws_bytes = p.gpu.workspace_bytes(1, 1, 4, 64)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    c = p.gpu.cache
    call = lambda **kw: kvq.kvq_decode_attn(
        kw.get("cache", c), kw.get("q", q), 1, kw.get("W", 1), kw.get("n_q", 4), ctx,
        kw.get("max_ctx", 64), p.bt, p.bt_host.shape[1], 0.1, kw.get("out", out),
        kw.get("ws", ws), kw.get("ws_bytes", ws_bytes))
    assert call() == kvq.KVQ_OK
    assert call(n_q=5) == kvq.KVQ_ERR_ARG
    assert call(ws_bytes=ws_bytes - 1) == kvq.KVQ_ERR_WORKSPACE
    nos = kvq.make_cache(kvq.KVQ_Q8, 2, 128, 16, p.gpu.n_blocks, p.gpu.k, p.gpu.v, None,
                         p.gpu.vs)
    assert call(cache=nos) == kvq.KVQ_ERR_ARG          # codes without scales: refused
    k = dev(np.zeros((1, 2, 128), np.float32))
    assert kvq.kvq_append(nos, k, k, 1, dev(np.zeros(1, np.int32)),
                          dev(np.zeros(1, np.int32)), p.bt, 1, p.bt_host.shape[1]) \
        == kvq.KVQ_ERR_ARG
    torch.cuda.synchronize()

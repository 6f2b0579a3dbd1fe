"""The cache file format on CPU: round trips and refusals.

Shaped after "Path F format v3: persist per-head INT8 KV scales for INT8 +
persistent KV interop" ("Scope": header, tokens, K/V body, scales body;
"Why": int8 codes without their scales must not be restored).
"""
import struct

import numpy as np
import pytest

from quantized_kv_cache_append_gb300 import KVQ_F16, KVQ_K8V4, KVQ_Q8
from quantized_kv_cache_append_gb300 import persist


def _arrays(fmt, n, n_kv, hd, seed):
    rng = np.random.default_rng(seed)
    if fmt == KVQ_F16:
        ck = rng.standard_normal((n, n_kv, hd)).astype(np.float16).view(np.uint16)
        cv = rng.standard_normal((n, n_kv, hd)).astype(np.float16).view(np.uint16)
        return ck, cv, None, None
    ck = rng.integers(-127, 128, (n, n_kv, hd)).astype(np.int8)
    sk = rng.random((n, n_kv, hd // 64)).astype(np.float16).view(np.uint16)
    if fmt == KVQ_K8V4:   # V: nibble bytes and one scale per 32 dims
        cv = rng.integers(0, 256, (n, n_kv, hd // 2)).astype(np.uint8)
        sv = rng.random((n, n_kv, hd // 32)).astype(np.float16).view(np.uint16)
        return ck, cv, sk, sv
    cv = rng.integers(-127, 128, (n, n_kv, hd)).astype(np.int8)
    sv = rng.random((n, n_kv, hd // 64)).astype(np.float16).view(np.uint16)
    return ck, cv, sk, sv


@pytest.mark.parametrize("fmt", [KVQ_F16, KVQ_Q8, KVQ_K8V4])
def test_round_trip(tmp_path, fmt):
    ck, cv, sk, sv = _arrays(fmt, 37, 3, 128, 1)
    tokens = np.arange(100, 137, dtype=np.int32)
    path = tmp_path / "c.kvq"
    persist.write_cells(path, fmt, 3, 128, tokens, ck, cv, sk, sv)
    t, ck2, cv2, sk2, sv2 = persist.read_cells(path, fmt, 3, 128)
    np.testing.assert_array_equal(t, tokens)
    np.testing.assert_array_equal(ck2, ck)
    np.testing.assert_array_equal(cv2, cv)
    if fmt != KVQ_F16:
        np.testing.assert_array_equal(sk2, sk)
        np.testing.assert_array_equal(sv2, sv)
    else:
        assert sk2 is None and sv2 is None
    raw = path.read_bytes()
    assert raw[:8] == b"KVQCELLS" and struct.unpack_from("<I", raw, 8)[0] == 3


def test_int8_without_scales_is_not_written(tmp_path):
    ck, cv, _, _ = _arrays(KVQ_Q8, 4, 1, 64, 2)
    with pytest.raises(persist.CacheFileError):
        persist.write_cells(tmp_path / "c.kvq", KVQ_Q8, 1, 64, None, ck, cv)


def _as_version2(path):
    """Rewrite a file as version 2: no scales body, scales_bytes 0."""
    raw = bytearray(path.read_bytes())
    fields = list(struct.unpack_from("<8sIIIIIIQQQ", raw))
    sbytes = fields[9]
    fields[1], fields[9] = 2, 0
    struct.pack_into("<8sIIIIIIQQQ", raw, 0, *fields)
    path.write_bytes(bytes(raw[: len(raw) - sbytes]))


def test_int8_pool_refuses_a_version2_file(tmp_path):
    path = tmp_path / "c.kvq"
    persist.write_cells(path, KVQ_Q8, 2, 64, None, *_arrays(KVQ_Q8, 9, 2, 64, 3))
    _as_version2(path)
    with pytest.raises(persist.CacheFileError, match="without their scales"):
        persist.read_cells(path, KVQ_Q8, 2, 64)


def test_fp16_pool_reads_a_version2_file(tmp_path):
    ck, cv, _, _ = _arrays(KVQ_F16, 9, 2, 64, 4)
    path = tmp_path / "c.kvq"
    persist.write_cells(path, KVQ_F16, 2, 64, None, ck, cv)
    _as_version2(path)
    _, ck2, cv2, _, _ = persist.read_cells(path, KVQ_F16, 2, 64)
    np.testing.assert_array_equal(ck2, ck)
    np.testing.assert_array_equal(cv2, cv)


@pytest.mark.parametrize("how", ["geometry", "format", "format_k8v4", "truncated", "magic",
                                 "version"])
def test_mismatched_or_damaged_files_are_refused(tmp_path, how):
    path = tmp_path / "c.kvq"
    persist.write_cells(path, KVQ_Q8, 2, 128, None, *_arrays(KVQ_Q8, 5, 2, 128, 5))
    fmt, n_kv, hd = KVQ_Q8, 2, 128
    if how == "geometry":
        n_kv = 4
    elif how == "format":
        fmt = KVQ_F16
    elif how == "format_k8v4":
        fmt = KVQ_K8V4
    elif how == "truncated":
        path.write_bytes(path.read_bytes()[:-7])
    elif how == "magic":
        raw = bytearray(path.read_bytes())
        raw[0:8] = b"NOTACACH"
        path.write_bytes(bytes(raw))
    else:
        raw = bytearray(path.read_bytes())
        struct.pack_into("<I", raw, 8, 9)
        path.write_bytes(bytes(raw))
    with pytest.raises(persist.CacheFileError):
        persist.read_cells(path, fmt, n_kv, hd)

"""The C ABI library builds, loads, exports exactly what include/kvq.h
declares, and its host-only parts behave (sizing, status strings, argument
validation).  No kernel is launched here: every call that could launch is
given one invalid argument that the host rejects first, and those calls are
skipped on a machine with a GPU (the GPU suite covers them with real
buffers)."""
import ctypes
import json
import os
import re
import subprocess

import pytest
import torch

import quantized_kv_cache_append_gb300 as kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "sizing_from_pages.json")


@pytest.fixture(scope="module")
def lib():
    kvq.build()
    return kvq.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^[A-Za-z_][\w \*]*?\b(kvq_\w+)\s*\(", text, flags=re.M)


def test_header_declarations_match_binding():
    assert tuple(_declared_functions()) == kvq.EXPORTED_SYMBOLS


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert getattr(lib, name) is not None
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    ours = sorted({ln.split()[-1] for ln in out.splitlines()
                   if ln.split()[-1].startswith("kvq_")})
    assert ours == sorted(_declared_functions())


def test_block_bytes_match_page_sizes(lib):
    g = json.load(open(GOLDEN))["kv_q8_pr"]
    cells, bs = g["cells"], 256
    n_kv, hd = 24, 256                       # 6144 K + 6144 V elements per cell
    per_block = lambda fmt: kvq.kvq_block_bytes(fmt, n_kv, hd, bs)
    gib = lambda fmt: per_block(fmt) * (cells // bs) / 2**30
    assert gib(kvq.KVQ_F16) == g["fp16_gib"]
    assert round(gib(kvq.KVQ_Q8), 1) == g["q8_gib"]
    assert per_block(kvq.KVQ_F16) == 2 * 2 * n_kv * hd * bs
    assert per_block(kvq.KVQ_Q8) == 2 * (n_kv * hd * bs + n_kv * hd * bs // 64 * 2)
    k8v4 = json.load(open(GOLDEN))["k8v4_pr"]["bytes_per_cell"]
    k_int8 = kvq.kvq_block_bytes(kvq.KVQ_Q8, 2, 256, 16) / 16 / 2     # K half, 512 dims
    assert k_int8 + 512 // 32 * 18 == k8v4
    assert kvq.kvq_block_bytes(kvq.KVQ_Q8, 1, 96, 16) == 0          # not a multiple of 64
    assert kvq.kvq_block_bytes(7, 1, 128, 16) == 0


def test_status_strings(lib):
    for s in range(5):
        assert kvq.kvq_status_string(s).startswith("KVQ_")
    assert "unknown" in kvq.kvq_status_string(99)


no_gpu_only = pytest.mark.skipif(torch.cuda.is_available(),
                                 reason="host-validation calls use fake addresses; "
                                        "covered with real buffers by the GPU suite")

FAKE = 1 << 20          # 256-byte aligned stand-in addresses, never dereferenced


def _cache(**kw):
    args = dict(fmt=kvq.KVQ_Q8, n_kv_heads=8, head_dim=128, block_size=256, n_blocks=4,
                k_data=FAKE, v_data=2 * FAKE, k_scales=3 * FAKE, v_scales=4 * FAKE)
    args.update(kw)
    return kvq.make_cache(args["fmt"], args["n_kv_heads"], args["head_dim"],
                          args["block_size"], args["n_blocks"], args["k_data"],
                          args["v_data"], args["k_scales"], args["v_scales"])


@no_gpu_only
@pytest.mark.parametrize("bad", [
    dict(k_scales=None), dict(v_scales=None),            # int8 codes without scales
    dict(head_dim=96), dict(block_size=48), dict(block_size=8), dict(fmt=3),
    dict(n_kv_heads=0), dict(k_data=FAKE + 16), dict(v_data=None),
])
def test_append_refuses_bad_cache(lib, bad):
    c = _cache(**bad)
    st = kvq.kvq_append(c, FAKE, FAKE, 4, FAKE, FAKE, FAKE, 1, 4, 0)
    assert st == kvq.KVQ_ERR_ARG


@no_gpu_only
def test_append_refuses_bad_arguments(lib):
    c = _cache()
    assert kvq.kvq_append(c, None, FAKE, 4, FAKE, FAKE, FAKE, 1, 4, 0) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_append(c, FAKE + 4, FAKE, 4, FAKE, FAKE, FAKE, 1, 4, 0) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_append(c, FAKE, FAKE, -1, FAKE, FAKE, FAKE, 1, 4, 0) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_append(c, FAKE, FAKE, 4, FAKE, FAKE, FAKE, 0, 4, 0) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_append(c, FAKE, FAKE, 0, None, None, None, 0, 0, 0) == kvq.KVQ_OK  # no-op


@no_gpu_only
def test_decode_refuses_bad_arguments(lib):
    c = _cache()
    def call(**kw):
        a = dict(q=FAKE, n_seq=1, W=1, n_q=32, ctx=FAKE, max_ctx=1024, bt=FAKE, mbps=4,
                 sm=0.088, out=FAKE, ws=FAKE, ws_bytes=1 << 30, cache=c)
        a.update(kw)
        return kvq.kvq_decode_attn(a["cache"], a["q"], a["n_seq"], a["W"], a["n_q"], a["ctx"],
                                   a["max_ctx"], a["bt"], a["mbps"], a["sm"], a["out"],
                                   a["ws"], a["ws_bytes"], 0)
    assert call(n_q=30) == kvq.KVQ_ERR_ARG                  # not a multiple of n_kv
    assert call(W=0) == kvq.KVQ_ERR_ARG
    assert call(W=17) == kvq.KVQ_ERR_ARG
    assert call(max_ctx=2048) == kvq.KVQ_ERR_ARG            # beyond the table width
    assert call(q=None) == kvq.KVQ_ERR_ARG
    assert call(out=FAKE + 8) == kvq.KVQ_ERR_ARG
    assert call(sm=float("nan")) == kvq.KVQ_ERR_ARG
    assert call(cache=_cache(v_scales=None)) == kvq.KVQ_ERR_ARG
    assert call(n_q=64, W=8) == kvq.KVQ_ERR_UNSUPPORTED     # 64 rows per KV head
    assert call(ws=None) == kvq.KVQ_ERR_WORKSPACE
    assert call(ws_bytes=16) == kvq.KVQ_ERR_WORKSPACE
    assert call(ws=FAKE + 64) == kvq.KVQ_ERR_WORKSPACE


@no_gpu_only
def test_compact_refuses_bad_arguments(lib):
    c = _cache()
    assert kvq.kvq_compact_f16(c, FAKE, 10, None, FAKE, 0) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_compact_f16(c, FAKE, -1, FAKE, FAKE, 0) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_compact_f16(_cache(k_scales=None), FAKE, 10, FAKE, FAKE, 0) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_compact_f16(c, None, 0, None, None, 0) == kvq.KVQ_OK   # no-op


def test_workspace_size_grows_with_context(lib):
    c = _cache()
    a = kvq.kvq_decode_workspace_bytes(c, 1, 1, 32, 1024)
    b = kvq.kvq_decode_workspace_bytes(c, 1, 1, 32, 32768)
    assert 0 < a <= b
    assert kvq.kvq_decode_workspace_bytes(c, 1, 1, 30, 1024) == 0


@no_gpu_only
def test_stream_fetch_refuses_mismatched_or_bad_arguments(lib):
    win = _cache(n_blocks=2)
    for bad in (dict(head_dim=256), dict(block_size=128), dict(n_kv_heads=4),
                dict(fmt=kvq.KVQ_F16), dict(k_scales=None), dict(k_data=FAKE + 16)):
        host = _cache(**bad)
        assert kvq.kvq_stream_fetch(host, win, FAKE, FAKE, 1, 0) == kvq.KVQ_ERR_ARG
    assert kvq.kvq_stream_fetch(_cache(), win, FAKE, FAKE, -1, 0) == kvq.KVQ_ERR_ARG
    # without a GPU no address is device-addressable: refused before any launch
    assert kvq.kvq_stream_fetch(_cache(), win, FAKE, FAKE, 1, 0) == kvq.KVQ_ERR_ARG


def test_missing_library_raises_instead_of_falling_back(tmp_path):
    # There is no CPU or library fallback: a missing libkvq.so is an error.
    with pytest.raises(RuntimeError, match="not built"):
        kvq.load_library(str(tmp_path / "libkvq.so"))


def test_failed_status_raises_with_its_name(lib):
    with pytest.raises(RuntimeError, match="kvq_append"):
        kvq.check(kvq.KVQ_ERR_ARG, "kvq_append")
    kvq.check(kvq.KVQ_OK, "kvq_append")   # success passes silently

"""Pin the cache formats' byte counts to the sizes the pages print.

#3084 qwen35 (FP16 K/V cache by default, int8 with --kv-q8), "Summary": at
262144 cells the FP32 cache is 12.0 GiB, FP16 6.0 GiB and the int8 form with
one FP16 scale per 64 dims 3.1 GiB.  12.0 GiB / 4 B / 262144 = 12288 K+V
elements per cell, so FP16 must cost 2 B and int8 1 + 2/64 B per element
(a 32-dim group or a 4-byte scale would print 3.2).  #711 kv (--kv k8v4
streams with --kv-resident), "What": INT8 K + Q4_0 V is 816 B per cell,
which for 512 dims is 512 * (1 + 2/64) + 512 * 18/32 -- the same int8 K part.
"""
import json
import os

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sizing_from_pages.json")


def _bytes_per_cell(fmt, n_kv, hd, parts=("k", "v", "ks", "vs")):
    bs = 16
    pool = oracle.PoolImage(fmt, n_kv, hd, bs, 1)
    total = sum(getattr(pool, p).nbytes for p in parts if getattr(pool, p) is not None)
    return total / bs


def test_oracle_pool_sizes_match_pages():
    g = json.load(open(GOLDEN))["kv_q8_pr"]
    cells = g["cells"]
    elems_per_cell = g["fp32_gib"] * 2**30 / 4 / cells          # K+V elements
    assert elems_per_cell == 12288
    n_kv, hd = 24, 256                                          # 6144 K dims per cell
    assert 2 * n_kv * hd == elems_per_cell
    gib = lambda fmt: _bytes_per_cell(fmt, n_kv, hd) * cells / 2**30
    assert gib(oracle.FMT_F16) == g["fp16_gib"]
    assert round(gib(oracle.FMT_Q8), 1) == g["q8_gib"]
    assert oracle.GROUP == g["q8_group_dims"]


def test_oracle_int8_k_part_matches_k8v4_cell():
    g = json.load(open(GOLDEN))["k8v4_pr"]
    k_part = _bytes_per_cell(oracle.FMT_Q8, 2, 256, parts=("k", "ks"))   # 512 K dims
    q4_0_v = 512 // 32 * 18
    assert k_part + q4_0_v == g["bytes_per_cell"]

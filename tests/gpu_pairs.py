"""Helpers for the GPU parity tests: run the same seeded inputs through the
CUDA library (via its C ABI) and through the CPU oracle, and compare.

Bars: cache bytes (codes, scales, fp16 values) and compaction bit-exact;
attention within max-abs 2e-3 and relative L2 1e-3 of the float64 oracle
evaluated on the oracle's own (bit-identical) cache.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import quantized_kv_cache_append_gb300 as kvq
from quantized_kv_cache_append_gb300.pool import PagedPool

MAX_ABS = 2e-3
REL_L2 = 1e-3

FORMATS = {"f16": (kvq.KVQ_F16, oracle.FMT_F16), "q8": (kvq.KVQ_Q8, oracle.FMT_Q8),
           "k8v4": (kvq.KVQ_K8V4, oracle.FMT_K8V4)}


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> numpy with the oracle's bit layout (fp16 as uint16)."""
    t = t.detach().cpu()
    if t.dtype == torch.float16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


class Pair:
    """A GPU pool and an oracle pool image fed the same appends."""

    def __init__(self, fmt_name, n_kv, head_dim, block_size, n_blocks, block_table):
        gfmt, ofmt = FORMATS[fmt_name]
        self.fmt_name = fmt_name
        self.gpu = PagedPool(gfmt, n_kv, head_dim, block_size, n_blocks)
        self.img = oracle.PoolImage(ofmt, n_kv, head_dim, block_size, n_blocks)
        self.bt_host = np.ascontiguousarray(block_table, dtype=np.int32)
        self.bt = dev(self.bt_host)

    def append(self, k, v, tok_seq, tok_pos):
        self.gpu.append(dev(k), dev(v), dev(np.asarray(tok_seq, np.int32)),
                        dev(np.asarray(tok_pos, np.int32)), self.bt)
        oracle.append(self.img, k, v, tok_seq, tok_pos, self.bt_host)

    def assert_cache_equal(self):
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(self.gpu.k), self.img.k), "K codes differ"
        assert np.array_equal(host_bits(self.gpu.v), self.img.v), "V codes differ"
        if self.fmt_name != "f16":
            assert np.array_equal(host_bits(self.gpu.ks), self.img.ks), "K scales differ"
            assert np.array_equal(host_bits(self.gpu.vs), self.img.vs), "V scales differ"

    def decode_gpu(self, q, ctx_lens, max_ctx, sm_scale):
        out = self.gpu.decode(dev(q), dev(np.asarray(ctx_lens, np.int32)), int(max_ctx),
                              self.bt, sm_scale)
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def decode_oracle(self, q, ctx_lens, sm_scale):
        return oracle.attention(self.img, q, ctx_lens, self.bt_host, sm_scale)

    def check_decode(self, q, ctx_lens, sm_scale, max_ctx=None):
        ctx = np.asarray(ctx_lens, np.int32)
        got = self.decode_gpu(q, ctx, int(ctx.max()) if max_ctx is None else max_ctx, sm_scale)
        ref = self.decode_oracle(q, ctx, sm_scale)
        assert_attention_close(got, ref)
        return got, ref

    def check_compact(self, seq, n_cells):
        row = self.bt_host[seq]
        ok, ov = self.gpu.compact(dev(row), n_cells)
        torch.cuda.synchronize()
        rk, rv = oracle.compact_f16(self.img, row, n_cells)
        assert np.array_equal(host_bits(ok), rk), "compacted K differs"
        assert np.array_equal(host_bits(ov), rv), "compacted V differs"


def attention_errors(got: np.ndarray, ref: np.ndarray):
    diff = got.astype(np.float64) - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_attention_close(got, ref):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite attention output"
    max_abs, rel = attention_errors(got, ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"max_abs={max_abs:.3g} rel_l2={rel:.3g}"

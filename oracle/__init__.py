"""Plain CPU oracle for the quantized K/V cache path (ctypes over kvq_oracle.c).

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's CPU
baseline leg may import this package; the product path (the CUDA library and
its Python binding) never does, and it shares no code with it.

Functions take and return numpy arrays in the layouts documented in
kvq_oracle.h.  fp16 values travel as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_HDR = os.path.join(_HERE, "kvq_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkvq_oracle.so")

FMT_F16 = 0
FMT_Q8 = 1
FMT_K8V4 = 2
GROUP = 64
Q4_BLOCK = 32

# No FMA contraction and no fast-math: float division, fabsf and rintf keep
# their IEEE meaning (round-to-nearest-even is the default mode).
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fno-strict-aliasing"]


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into a shared library (gcc); returns its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= newest_src):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_OMP_LIB_PATH = os.path.join(_BUILD_DIR, "libkvq_oracle_omp.so")


def build_parallel(force: bool = False):
    """The same source compiled with -fopenmp: kvo_attention then runs its
    independent (sequence, token, head) rows on OpenMP threads, each row with
    the same arithmetic as the single-threaded build.  Returns the library's
    path, or None when the compiler has no OpenMP support."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if (not force and os.path.exists(_OMP_LIB_PATH)
            and os.path.getmtime(_OMP_LIB_PATH) >= newest_src):
        return _OMP_LIB_PATH
    tmp = _OMP_LIB_PATH + f".tmp{os.getpid()}"
    r = subprocess.run(["gcc", *CFLAGS, "-fopenmp", "-o", tmp, _SRC, "-lm"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        return None
    os.replace(tmp, _OMP_LIB_PATH)
    return _OMP_LIB_PATH


def parallel_library(threads: int):
    """Path of the OpenMP build, set to use `threads` threads (None if it
    cannot be built).  Route attention() to it with use_library(path)."""
    path = build_parallel()
    if path is None:
        return None
    lib = _bind(ctypes.CDLL(path))
    lib.kvo_set_threads(int(threads))
    return path


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.kvo_fp16_from_float.restype = ctypes.c_uint16
    lib.kvo_fp16_from_float.argtypes = [ctypes.c_float]
    lib.kvo_fp16_to_float.restype = ctypes.c_float
    lib.kvo_fp16_to_float.argtypes = [ctypes.c_uint16]
    lib.kvo_fp16_from_float_array.restype = None
    lib.kvo_fp16_from_float_array.argtypes = [P, P, ctypes.c_int64]
    lib.kvo_fp16_to_float_array.restype = None
    lib.kvo_fp16_to_float_array.argtypes = [P, P, ctypes.c_int64]
    lib.kvo_quantize_row_q8.restype = I
    lib.kvo_quantize_row_q8.argtypes = [P, I, P, P]
    lib.kvo_quantize_row_q4r.restype = I
    lib.kvo_quantize_row_q4r.argtypes = [P, I, P, P]
    lib.kvo_hadamard_f32.restype = None
    lib.kvo_hadamard_f32.argtypes = [P, I]
    lib.kvo_append.restype = I
    lib.kvo_append.argtypes = [I, I, I, I, I, P, P, P, P, P, P, I, P, P, P, I]
    lib.kvo_attention.restype = I
    lib.kvo_attention.argtypes = [I, I, I, I, I, P, P, P, P, P, I, I, I, P, P, I,
                                  ctypes.c_float, P]
    lib.kvo_compact_f16.restype = I
    lib.kvo_compact_f16.argtypes = [I, I, I, I, I, P, P, P, P, P, I, P, P]
    lib.kvo_gather_cells.restype = I
    lib.kvo_gather_cells.argtypes = [I, I, I, I, I, P, P, P, P, P, I, P, P, P, P]
    lib.kvo_scatter_cells.restype = I
    lib.kvo_scatter_cells.argtypes = [I, I, I, I, I, P, P, P, P, P, I, P, P, P, P]
    lib.kvo_threads.restype = I
    lib.kvo_threads.argtypes = []
    lib.kvo_set_threads.restype = None
    lib.kvo_set_threads.argtypes = [I]
    lib.kvo_chunk_attention.restype = I
    lib.kvo_chunk_attention.argtypes = [I, I, I, P, P, P, I, I, ctypes.c_float, P]
    return lib


_lib = None
_override = None


def _load():
    global _lib
    if _override is not None:
        return _override
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


class use_library:
    """Context manager: route this module's functions to another build of
    kvq_oracle.c (the tests use it to run the pins against planted mistakes)."""

    def __init__(self, so_path: str):
        self._lib = _bind(ctypes.CDLL(so_path))

    def __enter__(self):
        global _override
        self._prev = _override
        _override = self._lib
        return self

    def __exit__(self, *exc):
        global _override
        _override = self._prev
        return False


def build_variant(src_text: str, out_dir: str, name: str) -> str:
    """Compile a (modified) copy of kvq_oracle.c with the oracle's flags."""
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, name + ".c")
    with open(src, "w") as f:
        f.write(src_text)
    so = os.path.join(out_dir, "lib" + name + ".so")
    subprocess.run(["gcc", *CFLAGS, "-I", _HERE, "-o", so, src, "-lm"], check=True)
    return so


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# fp16
# --------------------------------------------------------------------------

def fp16_bits(x) -> np.ndarray:
    """Round float32 values to IEEE binary16 (nearest, ties to even); bits."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().kvo_fp16_from_float_array(_ptr(x), _ptr(out), x.size)
    return out


def fp16_value(bits) -> np.ndarray:
    """Decode binary16 bit patterns to float32."""
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().kvo_fp16_to_float_array(_ptr(bits), _ptr(out), bits.size)
    return out


# --------------------------------------------------------------------------
# quantization
# --------------------------------------------------------------------------

def quantize_rows_q8(x):
    """Quantize rows of x [..., hd] -> (codes int8 [..., hd], scales uint16 [..., hd/64])."""
    x = _c(x, np.float32)
    hd = x.shape[-1]
    if hd % GROUP:
        raise ValueError("head_dim must be a multiple of 64")
    rows = x.reshape(-1, hd)
    codes = np.empty(rows.shape, dtype=np.int8)
    scales = np.empty((rows.shape[0], hd // GROUP), dtype=np.uint16)
    lib = _load()
    for i in range(rows.shape[0]):
        rc = lib.kvo_quantize_row_q8(_ptr(rows[i]), hd, _ptr(codes[i]), _ptr(scales[i]))
        if rc != 0:
            raise RuntimeError(f"kvo_quantize_row_q8 failed: {rc}")
    return codes.reshape(x.shape), scales.reshape(x.shape[:-1] + (hd // GROUP,))


def hadamard_f32(x):
    """Unnormalised Walsh-Hadamard transform of rows of x [..., n] in float32
    (the oracle's butterfly order); n a power of two."""
    x = _c(x, np.float32).copy()
    n = x.shape[-1]
    rows = x.reshape(-1, n)
    lib = _load()
    for i in range(rows.shape[0]):
        lib.kvo_hadamard_f32(_ptr(rows[i]), n)
    return rows.reshape(x.shape)


def quantize_rows_q4r(x):
    """K8V4's V rows: rotate, then Q4_0 per 32 rotated dims.  x [..., hd] ->
    (codes uint8 [..., hd/2] packed nibbles, scales uint16 [..., hd/32])."""
    x = _c(x, np.float32)
    hd = x.shape[-1]
    rows = x.reshape(-1, hd)
    codes = np.empty((rows.shape[0], hd // 2), dtype=np.uint8)
    scales = np.empty((rows.shape[0], hd // Q4_BLOCK), dtype=np.uint16)
    lib = _load()
    for i in range(rows.shape[0]):
        rc = lib.kvo_quantize_row_q4r(_ptr(rows[i]), hd, _ptr(codes[i]), _ptr(scales[i]))
        if rc != 0:
            raise RuntimeError(f"kvo_quantize_row_q4r failed: {rc}")
    return (codes.reshape(x.shape[:-1] + (hd // 2,)),
            scales.reshape(x.shape[:-1] + (hd // Q4_BLOCK,)))


def row_layout(fmt: int, head_dim: int):
    """(K element dtype, K elements per row, V dtype, V elements per row, K
    scales per row, V scales per row) of a pool row in each format."""
    if fmt == FMT_F16:
        return np.uint16, head_dim, np.uint16, head_dim, 0, 0
    if fmt == FMT_Q8:
        return np.int8, head_dim, np.int8, head_dim, head_dim // GROUP, head_dim // GROUP
    if fmt == FMT_K8V4:
        return np.int8, head_dim, np.uint8, head_dim // 2, head_dim // GROUP, head_dim // Q4_BLOCK
    raise ValueError(f"unknown format {fmt}")


# --------------------------------------------------------------------------
# paged cache image
# --------------------------------------------------------------------------

class PoolImage:
    """Host image of one layer's paged pool, in the library's layout."""

    def __init__(self, fmt: int, n_kv: int, head_dim: int, block_size: int, n_blocks: int):
        self.fmt, self.n_kv, self.head_dim = fmt, n_kv, head_dim
        self.block_size, self.n_blocks = block_size, n_blocks
        kdt, kn, vdt, vn, kng, vng = row_layout(fmt, head_dim)
        lead = (n_blocks, n_kv, block_size)
        self.k = np.zeros(lead + (kn,), dtype=kdt)
        self.v = np.zeros(lead + (vn,), dtype=vdt)
        self.ks = np.zeros(lead + (kng,), dtype=np.uint16) if kng else None
        self.vs = np.zeros(lead + (vng,), dtype=np.uint16) if vng else None

    def geometry(self):
        return (self.fmt, self.n_kv, self.head_dim, self.block_size, self.n_blocks)


def append(pool: PoolImage, k, v, tok_seq, tok_pos, block_table) -> None:
    """Quantize-on-write (or fp16 store) of n_tok new cells into the pool image."""
    k = _c(k, np.float32)
    v = _c(v, np.float32)
    tok_seq = _c(tok_seq, np.int32)
    tok_pos = _c(tok_pos, np.int32)
    bt = _c(block_table, np.int32)
    n_tok = tok_seq.shape[0]
    assert k.shape == (n_tok, pool.n_kv, pool.head_dim) and v.shape == k.shape
    rc = _load().kvo_append(*pool.geometry(), _ptr(pool.k), _ptr(pool.v),
                            _ptr(pool.ks), _ptr(pool.vs), _ptr(k), _ptr(v), n_tok,
                            _ptr(tok_seq), _ptr(tok_pos), _ptr(bt), bt.shape[1])
    if rc != 0:
        raise RuntimeError(f"kvo_append failed: {rc}")


def attention(pool: PoolImage, q, ctx_lens, block_table, sm_scale: float) -> np.ndarray:
    """float64 decode attention; q [n_seq][W][n_q][hd] -> out float64, same shape."""
    q = _c(q, np.float32)
    n_seq, W, n_q, hd = q.shape
    assert hd == pool.head_dim
    ctx = _c(ctx_lens, np.int32)
    bt = _c(block_table, np.int32)
    out = np.empty(q.shape, dtype=np.float64)
    rc = _load().kvo_attention(*pool.geometry(), _ptr(pool.k), _ptr(pool.v),
                               _ptr(pool.ks), _ptr(pool.vs), _ptr(q), n_seq, W, n_q,
                               _ptr(ctx), _ptr(bt), bt.shape[1], float(sm_scale),
                               _ptr(out))
    if rc != 0:
        raise RuntimeError(f"kvo_attention failed: {rc}")
    return out


def compact_f16(pool: PoolImage, block_table_row, n_cells: int):
    """Cells [0, n_cells) of one sequence -> (out_k, out_v) uint16 [n_kv][n_cells][hd]."""
    bt = _c(block_table_row, np.int32)
    out_k = np.empty((pool.n_kv, n_cells, pool.head_dim), dtype=np.uint16)
    out_v = np.empty_like(out_k)
    rc = _load().kvo_compact_f16(*pool.geometry(), _ptr(pool.k), _ptr(pool.v),
                                 _ptr(pool.ks), _ptr(pool.vs), _ptr(bt), n_cells,
                                 _ptr(out_k), _ptr(out_v))
    if rc != 0:
        raise RuntimeError(f"kvo_compact_f16 failed: {rc}")
    return out_k, out_v


def chunk_attention(k16, v16, q, sm_scale: float) -> np.ndarray:
    """float64 prompt-chunk attention over fp16 staging.

    k16, v16: uint16 fp16 bits [n_kv][P][hd]; q float32 [T][n_q][hd] (the
    chunk's tokens are the last T cells; token t sees cells [0, P - T + t]).
    Returns float64 [T][n_q][hd]."""
    k16 = _c(k16, np.uint16)
    v16 = _c(v16, np.uint16)
    q = _c(q, np.float32)
    n_kv, P, hd = k16.shape
    T, n_q, qhd = q.shape
    assert qhd == hd and v16.shape == k16.shape
    out = np.empty(q.shape, dtype=np.float64)
    rc = _load().kvo_chunk_attention(n_kv, P, hd, _ptr(k16), _ptr(v16), _ptr(q), T, n_q,
                                     float(sm_scale), _ptr(out))
    if rc != 0:
        raise RuntimeError(f"kvo_chunk_attention failed: {rc}")
    return out


def gather_cells(pool: PoolImage, block_table_row, n_cells: int):
    """Cells [0, n_cells) of one sequence, token-major: (codes_k, codes_v,
    scales_k, scales_v) with codes [n_cells][n_kv][hd] (uint16 fp16 bits or
    int8) and scales [n_cells][n_kv][hd/64] uint16 (None for fp16); K8V4's V
    codes are uint8 [..][hd/2] and its V scales [..][hd/32]."""
    bt = _c(block_table_row, np.int32)
    kdt, kn, vdt, vn, kng, vng = row_layout(pool.fmt, pool.head_dim)
    ck = np.empty((n_cells, pool.n_kv, kn), dtype=kdt)
    cv = np.empty((n_cells, pool.n_kv, vn), dtype=vdt)
    sk = np.empty((n_cells, pool.n_kv, kng), dtype=np.uint16) if kng else None
    sv = np.empty((n_cells, pool.n_kv, vng), dtype=np.uint16) if vng else None
    rc = _load().kvo_gather_cells(*pool.geometry(), _ptr(pool.k), _ptr(pool.v), _ptr(pool.ks),
                                  _ptr(pool.vs), _ptr(bt), n_cells, _ptr(ck), _ptr(cv),
                                  _ptr(sk), _ptr(sv))
    if rc != 0:
        raise RuntimeError(f"kvo_gather_cells failed: {rc}")
    return ck, cv, sk, sv


def scatter_cells(pool: PoolImage, block_table_row, codes_k, codes_v, scales_k=None,
                  scales_v=None) -> None:
    """Write token-major cells back into the pool (the inverse of gather_cells)."""
    bt = _c(block_table_row, np.int32)
    kdt, _, vdt, _, _, _ = row_layout(pool.fmt, pool.head_dim)
    ck, cv = _c(codes_k, kdt), _c(codes_v, vdt)
    sk = None if scales_k is None else _c(scales_k, np.uint16)
    sv = None if scales_v is None else _c(scales_v, np.uint16)
    rc = _load().kvo_scatter_cells(*pool.geometry(), _ptr(pool.k), _ptr(pool.v), _ptr(pool.ks),
                                   _ptr(pool.vs), _ptr(bt), ck.shape[0], _ptr(ck), _ptr(cv),
                                   _ptr(sk), _ptr(sv))
    if rc != 0:
        raise RuntimeError(f"kvo_scatter_cells failed: {rc}")

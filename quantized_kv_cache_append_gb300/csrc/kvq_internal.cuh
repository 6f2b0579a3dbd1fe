// kvq_internal.cuh -- internal declarations shared by the library's
// translation units (not part of the C ABI; see include/kvq.h).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"
#include "kvq_context_cache.h"

namespace kvq {

constexpr int kGroup = KVQ_GROUP;  // dims per fp16 scale in the int8 format
constexpr int kQ4Block = KVQ_Q4_BLOCK;  // rotated V dims per fp16 scale in K8V4
constexpr uint32_t kDefaultWaitLimit = 1u << 25;  // polls of a copy wait before it is lost

// Walsh-Hadamard transform (Sylvester order, no normalisation) of a row of
// 32 * U * NI values held by one warp: lane l holds x[i][e] = dim e + U l +
// 32 U i (units of U consecutive dims, the lanes' units side by side, NI
// such runs).  The stages run h = 1, 2, ..., 16 U NI: those below U inside
// a unit, those up to 16 U between lanes l and l ^ (h / U), the rest
// between a lane's units.  Each stage turns dims (j, j + h), bit h of j
// clear, into (x_j + x_{j+h}, x_j - x_{j+h}), so every fp32 sum and
// difference is the one the stage-by-stage definition rounds.
template <int U, int NI>
__device__ __forceinline__ void wht_warp(float (&x)[NI][U], int lane) {
#pragma unroll
  for (int h = 1; h < U; h *= 2)
#pragma unroll
    for (int i = 0; i < NI; ++i)
#pragma unroll
      for (int e = 0; e < U; ++e)
        if (!(e & h)) {
          const float a = x[i][e], b = x[i][e + h];
          x[i][e] = __fadd_rn(a, b);
          x[i][e + h] = __fsub_rn(a, b);
        }
#pragma unroll
  for (int hl = 1; hl < 32; hl *= 2) {
    // the lower lane keeps x + y, the upper y - x: fma(x, +-1, y), whose
    // product is exact, rounds the same sum or difference once
    const float sgn = (lane & hl) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i)
#pragma unroll
      for (int e = 0; e < U; ++e) {
        const float y = __shfl_xor_sync(0xffffffffu, x[i][e], hl);
        x[i][e] = __fmaf_rn(x[i][e], sgn, y);
      }
  }
#pragma unroll
  for (int hi = 1; hi < NI; hi *= 2)
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (!(i & hi))
#pragma unroll
        for (int e = 0; e < U; ++e) {
          const float a = x[i][e], b = x[i + hi][e];
          x[i][e] = __fadd_rn(a, b);
          x[i + hi][e] = __fsub_rn(a, b);
        }
}

// Walsh-Hadamard transform of a row held by LPR lanes of VPL consecutive
// dims each: stages h = 1 .. VPL/2 inside a lane, then h = VPL .. HD/2
// between lanes j and j ^ (h / VPL) of the group (its lanes are an aligned
// run, so the partner stays inside it).  Each stage turns dims (i, i + h),
// bit h of i clear, into (x_i + x_{i+h}, x_i - x_{i+h}), every sum and
// difference rounded once in fp32, as the stage-by-stage definition does
// (the upper lane's y - x as fma(x, -1, y), an exact product).
template <int VPL, int LPR>
__device__ __forceinline__ void wht_group(float (&x)[VPL], int lane) {
#pragma unroll
  for (int h = 1; h < VPL; h *= 2)
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (!(i & h)) {
        const float p = x[i], q = x[i + h];
        x[i] = __fadd_rn(p, q);
        x[i + h] = __fsub_rn(p, q);
      }
#pragma unroll
  for (int hl = 1; hl < LPR; hl *= 2) {
    const float sgn = (lane & hl) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const float y = __shfl_xor_sync(0xffffffffu, x[i], hl);
      x[i] = __fmaf_rn(x[i], sgn, y);
    }
  }
}

// ---------------------------------------------------------------------------
// Pool geometry as the kernels see it.
// ---------------------------------------------------------------------------
struct Pool {
  const void* k;       // codes: fp16 or int8 [n_blocks][n_kv][bs][hd]
  const void* v;       // (K8V4: V nibbles [n_blocks][n_kv][bs][hd/2])
  const __half* ks;    // scales: fp16 [n_blocks][n_kv][bs][hd/64] (int8 only)
  const __half* vs;    // (K8V4: V scales [n_blocks][n_kv][bs][hd/32])
  int n_kv;
  int bs_log2;         // block size = 1 << bs_log2
  int n_blocks;
};

struct AppendArgs {
  void* k_dst;
  void* v_dst;
  __half* ks_dst;
  __half* vs_dst;
  const float* k;      // [n_tok][n_kv][hd]
  const float* v;
  const int32_t* tok_seq;
  const int32_t* tok_pos;
  const int32_t* block_table;
  int n_tok, n_kv, bs_log2, n_blocks, n_seq, max_blocks;
};

// Split plan of one decode call: the context of every (sequence, KV head)
// is cut into nsplit ranges of split_cells cells; each range is one CTA of
// the partial kernel.
struct DecodePlan {
  int use_mma;         // 1: the tensor-core kernels can run (their setup succeeded)
  int rows;            // R = G * W query rows per (sequence, KV head)
  int rt_rows;         // rows per CTA (R, or the widest row tile the head dim allows)
  int n_rt;            // row tiles per work item: ceil(R / rt_rows)
  int split_cells;     // cells per split (a multiple of the cell tile)
  int nsplit;          // splits per (sequence, KV head), one partial each
  size_t off_o, off_ml, bytes;  // workspace layout
};

// Division of a 32-bit x by a divisor d fixed per call: q = x / d is the
// high 64 bits of x * ceil(2^64 / d), exact for every x < 2^64 / d, so for
// every 32-bit x (d = 1 keeps m = 0 and q = x).  Built on the host; on the
// device one multiply replaces the instruction sequence of a division by a
// run-time value.
struct FastDiv {
  unsigned long long m;
  unsigned d;
};

inline FastDiv make_fastdiv(unsigned d) {
  FastDiv f;
  f.d = d;
  f.m = d <= 1 ? 0ull : ~0ull / d + 1ull;
  return f;
}

#ifdef __CUDACC__
__device__ __forceinline__ unsigned fdiv(unsigned x, const FastDiv& f) {
  return f.d <= 1 ? x : (unsigned)__umul64hi((unsigned long long)x, f.m);
}
#endif

struct DecodeArgs {
  Pool pool;
  const float* q;      // [n_seq][W][n_q][hd]
  float* out;          // [n_seq][W][n_q][hd]
  const int32_t* ctx_lens;
  const int32_t* block_table;
  float* ws_o;         // [n_seq][n_kv][nsplit][R][hd]   unnormalised partial outputs
  float* ws_ml;        // [n_seq][n_kv][nsplit][R][2]    (running max, sum), log2 domain
  int n_seq, W, n_q, G, R, max_blocks, split_cells, nsplit;
  int RT, n_rt;        // query rows per CTA and CTAs (row tiles) per work item
  unsigned long long g_magic;  // ceil(2^32 / G): (r * g_magic) >> 32 == r / G for
                               // every row index r < 2^32 / G (rows are < 32)
  FastDiv div_nkv, div_nrt, div_split;  // n_kv, n_rt, split_cells
  float qscale;        // sm_scale * log2(e): logits come out in the log2 domain
  uint32_t wait_limit; // polls of a copy wait before it is declared lost
  uint32_t extra_tx;   // bytes added to each stage's expected count (0; >0 only
                       // in the failure-path test, where no copy delivers them)
};

struct CompactArgs {
  Pool pool;
  const int32_t* block_row;
  int n_cells;
  __half* out_k;       // [n_kv][n_cells][hd]
  __half* out_v;
};

// A sequence's cells between the pool and token-major runs (kvq_persist.cu).
struct PersistArgs {
  Pool pool;               // the pool, read by the gather
  void* pool_k;            // the same arrays, written by the scatter
  void* pool_v;
  __half* pool_ks;
  __half* pool_vs;
  const int32_t* block_row;
  int n_cells;
  void* codes_k;           // [n_cells][n_kv][hd]: written by gather, read by scatter
  void* codes_v;           // (K8V4: [n_cells][n_kv][hd/2] nibbles)
  __half* scales_k;        // [n_cells][n_kv][hd/64] (int8 and K8V4)
  __half* scales_v;        // (K8V4: [n_cells][n_kv][hd/32])
};

// Launchers (host side, one per translation unit).  They return the launch
// status from the runtime.
cudaError_t launch_append(int fmt, int hd, const AppendArgs& a, cudaStream_t s);
cudaError_t launch_compact(int fmt, int hd, const CompactArgs& a, cudaStream_t s);
cudaError_t launch_persist(int fmt, int hd, bool gather, const PersistArgs& a, cudaStream_t s);

// Split-K decode (kvq_decode_mma.cu): shapes it covers, its cell tile, the
// query rows one CTA holds, resident CTAs per SM of the kernel serving a
// row count (0 if unavailable), and its launcher (partial + combine).
bool mma_decode_supported(int fmt, int hd, int rows);
int mma_cell_tile();
int mma_rows_per_cta(int hd);
int mma_ctas_per_sm(int fmt, int hd, int rows);
cudaError_t launch_decode_mma_partial(int fmt, int hd, const DecodePlan& p, const DecodeArgs& a,
                                      cudaStream_t s);

// The driver's cuTensorMapEncodeTiled (version 12000), looked up once; null
// if the driver does not provide it.
void* tensor_map_encoder();

// Identity of the CUDA context current on the calling thread (cuCtxGetId),
// 0 if none is current or the driver cannot say.  Kernel attributes, module
// symbols and occupancy belong to a context: a process that drives several
// devices, or that resets one (cudaDeviceReset makes a new context), needs
// its one-time kernel setup redone for the new context.
unsigned long long current_context_id();

// One-time setup of a ContextCache (kvq_context_cache.h) for the current
// device and context: `setup(T*) -> bool` runs when the device's slot was
// filled under another context (or never); a failed setup leaves no sticky
// runtime status behind.
template <class T, class F>
bool per_context(ContextCache<T>& cache, T* out, F setup) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return cache.get(dev, current_context_id(), out,
                   [&](T* v) {
                     if (setup(v)) return true;
                     (void)cudaGetLastError();
                     return false;
                   },
                   [] { return current_context_id(); });
}

// Block streaming (kvq_stream.cu): the residency plan (host only) and the
// fetch of blocks from the host copy into window slots.
kvq_status stream_plan(int n_host_blocks, int n_slots, int32_t* slot_of_block, int32_t* block_of_slot,
                       int64_t* last_use, int64_t* clock, const int32_t* block_table, int n_seq,
                       int max_blocks, const int32_t* ctx_lens, int block_size, int32_t* slot_table,
                       int32_t* fetch_src, int32_t* fetch_dst, int* n_fetch, int* n_hits);
cudaError_t launch_fetch(int fmt, int hd, const kvq_cache* host, const kvq_cache* win,
                         const int32_t* fetch_src, const int32_t* fetch_dst, int n_fetch,
                         cudaStream_t s);

// Prompt-chunk attention over fp16 staging (kvq_chunk.cu).
struct ChunkArgs {
  const __half* k16;   // [n_kv][P][hd]
  const __half* v16;
  const float* q;      // [T][n_q][hd]
  float* out;          // [T][n_q][hd]
  int n_kv, P, T, n_q, G;
  float qscale;        // sm_scale * log2(e)
  uint32_t wait_limit; // polls of an mbarrier wait before it is declared lost
  uint32_t extra_tx;   // bytes added to each K / V stage's expected count (0; >0 only
                       // in the lost-wait test, which makes every copy wait run out)
};
cudaError_t launch_chunk_attn(int hd, const ChunkArgs& a, cudaStream_t s);

}  // namespace kvq

// kvq_internal.cuh -- internal declarations shared by the library's
// translation units (not part of the C ABI; see include/kvq.h).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

constexpr int kGroup = KVQ_GROUP;  // dims per fp16 scale in the int8 format

// ---------------------------------------------------------------------------
// Pool geometry as the kernels see it.
// ---------------------------------------------------------------------------
struct Pool {
  const void* k;       // codes: fp16 or int8 [n_blocks][n_kv][bs][hd]
  const void* v;
  const __half* ks;    // scales: fp16 [n_blocks][n_kv][bs][hd/64] (int8 only)
  const __half* vs;
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
  int use_mma;         // 1: tensor-core partial kernel (kvq_decode_mma.cu)
  int rows;            // R = G * W query rows per (sequence, KV head)
  int rows_pad;        // R rounded up to the kernel's row tile
  int split_cells;     // cells per split (a multiple of the cell tile)
  int nsplit;          // splits per (sequence, KV head), one partial each
  size_t off_o, off_ml, bytes;  // workspace layout
};

struct DecodeArgs {
  Pool pool;
  const float* q;      // [n_seq][W][n_q][hd]
  float* out;          // [n_seq][W][n_q][hd]
  const int32_t* ctx_lens;
  const int32_t* block_table;
  float* ws_o;         // [n_seq][n_kv][nsplit][R][hd]   unnormalised partial outputs
  float* ws_ml;        // [n_seq][n_kv][nsplit][R][2]    (running max, sum), log2 domain
  int n_seq, W, n_q, G, R, max_blocks, split_cells, nsplit;
  float qscale;        // sm_scale * log2(e): logits come out in the log2 domain
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
  void* codes_v;
  __half* scales_k;        // [n_cells][n_kv][hd/64] (int8 only)
  __half* scales_v;
};

// Launchers (host side, one per translation unit).  They return the launch
// status from the runtime.
cudaError_t launch_append(int fmt, int hd, const AppendArgs& a, cudaStream_t s);
cudaError_t launch_compact(int fmt, int hd, const CompactArgs& a, cudaStream_t s);
cudaError_t launch_persist(int fmt, int hd, bool gather, const PersistArgs& a, cudaStream_t s);
bool decode_supported(int fmt, int hd, int rows);
int decode_rows_pad(int hd, int rows);
int decode_cell_tile();
cudaError_t launch_decode(int fmt, int hd, const DecodePlan& plan, const DecodeArgs& a,
                          cudaStream_t s);

// Tensor-core partial kernel (kvq_decode_mma.cu): shapes it covers, its cell
// tile, resident CTAs per SM (0 if unavailable), and its launcher (partial +
// combine).
bool mma_decode_supported(int fmt, int hd, int rows);
int mma_cell_tile();
int mma_ctas_per_sm(int fmt, int hd, int rows);
cudaError_t launch_decode_mma_partial(int fmt, int hd, const DecodePlan& p, const DecodeArgs& a,
                                      cudaStream_t s);

// The driver's cuTensorMapEncodeTiled (version 12000), looked up once; null
// if the driver does not provide it.
void* tensor_map_encoder();

// Prompt-chunk attention over fp16 staging (kvq_chunk.cu).
struct ChunkArgs {
  const __half* k16;   // [n_kv][P][hd]
  const __half* v16;
  const float* q;      // [T][n_q][hd]
  float* out;          // [T][n_q][hd]
  int n_kv, P, T, n_q, G;
  float qscale;        // sm_scale * log2(e)
};
cudaError_t launch_chunk_attn(int hd, const ChunkArgs& a, cudaStream_t s);

}  // namespace kvq

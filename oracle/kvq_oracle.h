/*
 * kvq_oracle.h -- plain CPU oracle for the quantized K/V cache path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this code: only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only on the same seeded inputs.
 *
 * Everything here is scalar C, written to be read against its sources:
 *   [kv-q8 PR]  "#3084 qwen35: FP16 K/V cache by default, int8 with --kv-q8
 *               (262144 fits a 16 GiB card)" -- sections "Summary",
 *               "What changed", "Extra Notes".
 *   [k8v4 PR]   "#711 kv: --kv k8v4 streams with --kv-resident" -- section
 *               "How" (a block moved as byte runs: codes, then scales).
 *
 * Layouts (all row-major, element = one K or V value):
 *   pool codes   [n_blocks][n_kv][block_size][head_dim]   fp16 bits or int8
 *   pool scales  [n_blocks][n_kv][block_size][head_dim/64] fp16 bits (int8 only)
 *   q, out       [n_seq][W][n_q][head_dim]
 *   new k, v     [n_tok][n_kv][head_dim]
 *   block table  [n_seq][max_blocks_per_seq]
 * Logical cell p of sequence b lives in block table[b][p / block_size],
 * slot p % block_size.
 *
 * Return value of the int functions: 0 on success, a negative number when an
 * argument or an index is out of range (nothing is written in that case for
 * the failing row; the caller treats it as a test failure).
 */
#ifndef KVQ_ORACLE_H
#define KVQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVO_FMT_F16 0
#define KVO_FMT_Q8 1
#define KVO_FMT_K8V4 2 /* int8 K (as KVO_FMT_Q8) + rotated Q4_0 V */
#define KVO_GROUP 64
#define KVO_Q4_BLOCK 32

/* IEEE-754 binary16 conversion, round to nearest, ties to even, subnormals
 * kept, overflow to infinity. */
uint16_t kvo_fp16_from_float(float x);
float kvo_fp16_to_float(uint16_t h);
void kvo_fp16_from_float_array(const float *x, uint16_t *out, int64_t n);
void kvo_fp16_to_float_array(const uint16_t *h, float *out, int64_t n);

/* Quantize one row of hd values: per group of 64 dims one fp16 scale
 * s = fp16(max|x| / 127) and codes clamp(rint(x / s), -127, 127). */
int kvo_quantize_row_q8(const float *x, int hd, int8_t *codes, uint16_t *scales);

/* In-place Walsh-Hadamard transform of n values (n a power of two), fp32:
 * stages h = 1, 2, 4, ..., n/2; in each, every pair (j, j + h) with bit h of
 * j clear becomes (x[j] + x[j+h], x[j] - x[j+h]).  No normalisation: applied
 * twice it multiplies by n. */
void kvo_hadamard_f32(float *x, int n);

/* K8V4's V row: the row rotated by the Walsh-Hadamard transform, then
 * Q4_0 per block of 32 rotated dims: d = fp16(m / -8) with m the block's
 * element of largest magnitude (the first on ties), code = clamp(rint(y /
 * d), -8, 7) + 8 (0..15; 8 when d is 0), value (code - 8) * d.  codes[j]
 * holds dims 2j (low nibble) and 2j + 1 (high nibble); one fp16 d per 32
 * dims. */
int kvo_quantize_row_q4r(const float *x, int hd, uint8_t *codes, uint16_t *scales);

/* Write n_tok new cells (K and V) into the paged pool image.  KVO_FMT_K8V4:
 * v_data is [n_blocks][n_kv][block_size][hd/2] packed nibbles and v_scales
 * [..][hd/32]. */
int kvo_append(int fmt, int n_kv, int hd, int block_size, int n_blocks,
               void *k_data, void *v_data, uint16_t *k_scales, uint16_t *v_scales,
               const float *k, const float *v, int n_tok,
               const int32_t *tok_seq, const int32_t *tok_pos,
               const int32_t *block_table, int max_blocks_per_seq);

/* Decode attention in float64 over the dequantized pool.  Query token w of
 * sequence b sees cells [0, ctx_lens[b] - W + w]; query head h reads KV head
 * h / (n_q / n_kv).  A query with no visible cell gets an all-zero output. */
int kvo_attention(int fmt, int n_kv, int hd, int block_size, int n_blocks,
                  const void *k_data, const void *v_data,
                  const uint16_t *k_scales, const uint16_t *v_scales,
                  const float *q, int n_seq, int W, int n_q,
                  const int32_t *ctx_lens, const int32_t *block_table,
                  int max_blocks_per_seq, float sm_scale, double *out);

/* Threads kvo_attention spreads its rows over: 1, or the OpenMP thread
 * count of a build made with -fopenmp (the multi-core CPU baseline). */
int kvo_threads(void);
void kvo_set_threads(int n);

/* Copy cells [0, n_cells) of one sequence out to contiguous fp16
 * out_k/out_v [n_kv][n_cells][hd] (fp16 bits). */
int kvo_compact_f16(int fmt, int n_kv, int hd, int block_size, int n_blocks,
                    const void *k_data, const void *v_data,
                    const uint16_t *k_scales, const uint16_t *v_scales,
                    const int32_t *block_table_row, int n_cells,
                    uint16_t *out_k, uint16_t *out_v);

/* Persistence: cells [0, n_cells) of one sequence gathered out of the pool
 * into token-major runs, and scattered back.  codes_k / codes_v are
 * [n_cells][n_kv][hd] elements of the pool's format (fp16 bits or int8);
 * scales_k / scales_v [n_cells][n_kv][hd/64] fp16 bits, required for int8
 * (-2 without them) and ignored for fp16.  K8V4: codes_v [..][hd/2] packed
 * nibbles and scales_v [..][hd/32], both required. */
int kvo_gather_cells(int fmt, int n_kv, int hd, int block_size, int n_blocks,
                     const void *k_data, const void *v_data,
                     const uint16_t *k_scales, const uint16_t *v_scales,
                     const int32_t *block_table_row, int n_cells,
                     void *codes_k, void *codes_v, uint16_t *scales_k, uint16_t *scales_v);
int kvo_scatter_cells(int fmt, int n_kv, int hd, int block_size, int n_blocks,
                      void *k_data, void *v_data, uint16_t *k_scales, uint16_t *v_scales,
                      const int32_t *block_table_row, int n_cells,
                      const void *codes_k, const void *codes_v,
                      const uint16_t *scales_k, const uint16_t *scales_v);

/* Attention of a prompt chunk over contiguous fp16 staging, float64.  The
 * staging k16/v16 [n_kv][P][hd] (fp16 bits) holds the sequence's P cells;
 * the chunk's T query tokens are its last T cells, so token t sees cells
 * [0, P - T + t].  q and out are [T][n_q][hd]; query head h reads KV head
 * h / (n_q / n_kv). */
int kvo_chunk_attention(int n_kv, int P, int hd, const uint16_t *k16, const uint16_t *v16,
                        const float *q, int T, int n_q, float sm_scale, double *out);

#ifdef __cplusplus
}
#endif
#endif

/*
 * kvq.h -- C ABI of the quantized K/V cache library (one GB300, sm_103a).
 *
 * The library keeps a transformer's K/V cache in a paged pool, as FP16, as
 * int8 codes with one FP16 scale per 64 head dims, or as K8V4 (int8 K and
 * rotated 4-bit V), and runs the calls that touch it on the decode / verify
 * / prompt paths:
 *
 *   kvq_append       quantize-on-write of new K/V rows into the pool
 *   kvq_decode_attn  GQA attention of 1..W query tokens against the pool,
 *                    as split-K partials merged by a log-sum-exp combine
 *   kvq_compact_f16  the pool copied out to contiguous FP16 staging
 *   kvq_chunk_attn   attention of a prompt chunk over that staging
 *   kvq_gather_cells / kvq_scatter_cells
 *                    a sequence's codes and scales out of / into the pool
 *   kvq_stream_plan / kvq_stream_fetch
 *                    a resident window of device blocks over a host copy
 *
 * Sources (page title, section):
 *   [kv-q8 PR]  "#3084 qwen35: FP16 K/V cache by default, int8 with --kv-q8
 *               (262144 fits a 16 GiB card)": "Summary" (the two formats,
 *               one FP16 scale per 64 dims), "What changed" (the formula
 *               scale = fp16(max|x|/127), code = clamp(rint(x/scale),
 *               -127, 127); k_attn_prep / k_attn_part / k_kv_f16 templated on
 *               the cache format; scale arrays carried beside the code
 *               arrays), "Extra Notes" (split-K decode; k_kv_f16 compacts
 *               [kvh][ctx][HD] into [kvh][P][HD] halves for the prompt).
 *   [k8v4 PR]   "#711 kv: --kv k8v4 streams with --kv-resident": "How"
 *               (a block is a list of byte runs -- codes, then scales; the
 *               decode, verify-window and prompt appends; a writer that
 *               tests one pointer and silently skips the other), "Tests"
 *               (the negative control that catches that skip), "What"
 *               (K8V4: INT8 K + rotated Q4_0 V, 816 B per cell).
 *   [Path F v3] "Path F format v3: persist per-head INT8 KV scales for
 *               INT8 + persistent KV interop": "Why", "Scope" (int8 bytes
 *               without their scales are refused, not used).
 *
 * Conventions for every call
 *   - All device arrays are owned and allocated by the caller; the library
 *     allocates nothing and keeps no state between calls beyond one-time
 *     kernel setup (each kernel configuration's shared-memory limit and
 *     occupancy, kept per device and redone when that device's context
 *     changes, so one process may drive several devices) and
 *     kvq_decode_attn_static's scratch.  Pointers marked "device" must be
 *     device (or managed) memory of the current device.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  No call reads device memory on the host or
 *     synchronizes.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid argument returns KVQ_ERR_ARG (or KVQ_ERR_UNSUPPORTED for a
 *     valid but unimplemented shape) and launches nothing.  No call aborts,
 *     exits, throws or traps on the device.  A launch failure reported by
 *     the runtime returns KVQ_ERR_CUDA.
 *   - Device-side preconditions (not checked on the host, since the values
 *     live on the device): block ids in the block table lie in
 *     [0, n_blocks) for every cell that is read or written; token positions
 *     are < max_blocks_per_seq * block_size; 0 <= ctx_lens[b] <= max_ctx (a
 *     query token with no visible cell, as when ctx_lens[b] < W, gets 0).
 *     Breaking them gives unspecified values for the cells involved but no
 *     out-of-bounds access: every kernel checks each block id it reads
 *     against [0, n_blocks) and skips (append, compaction) or reads as
 *     zeros (attention) a cell whose id is out of range; the append kernel
 *     checks tok_seq against [0, n_seq) and tok_pos against the table width;
 *     the attention kernels clamp ctx_lens[b] to [0, max_blocks_per_seq *
 *     block_size].
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Cache formats ([kv-q8 PR], "Summary"). */
typedef enum {
    KVQ_F16 = 0, /* K and V stored as IEEE fp16 (round to nearest even)      */
    KVQ_Q8 = 1,  /* int8 codes + one fp16 scale per 64 dims of a row         */
    KVQ_K8V4 = 2 /* K as KVQ_Q8; V rotated (Walsh-Hadamard), then 4-bit      */
                 /* codes + one fp16 scale per 32 rotated dims ([k8v4 PR])  */
} kvq_format;

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_ARG = 1,         /* null / misaligned pointer, bad size or shape  */
    KVQ_ERR_UNSUPPORTED = 2, /* valid request outside the implemented shapes */
    KVQ_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required   */
    KVQ_ERR_CUDA = 4         /* the CUDA runtime reported a launch error     */
} kvq_status;

/* Group of head dims sharing one fp16 scale in KVQ_Q8 (and K8V4's K). */
#define KVQ_GROUP 64
/* Block of rotated V dims sharing one fp16 scale in KVQ_K8V4. */
#define KVQ_Q4_BLOCK 32

/*
 * One layer's paged K/V pool.  A physical block holds block_size consecutive
 * cells of one sequence for all n_kv_heads KV heads; K and V, codes and
 * scales are four separate arrays ("byte runs", [k8v4 PR] "How"):
 *
 *   k_data, v_data     [n_blocks][n_kv_heads][block_size][head_dim]
 *                      fp16 (KVQ_F16) or int8 (KVQ_Q8)
 *   k_scales, v_scales [n_blocks][n_kv_heads][block_size][head_dim / 64]
 *                      fp16 bits; KVQ_Q8 only (must be NULL-free for Q8,
 *                      ignored for F16)
 *
 * KVQ_K8V4 keeps K as KVQ_Q8 does (k_data int8, k_scales per 64 dims) and V
 * as two other runs:
 *
 *   v_data             [n_blocks][n_kv_heads][block_size][head_dim / 2]
 *                      bytes: two 4-bit codes each, dim 2j in the low
 *                      nibble of byte j, dim 2j + 1 in the high nibble
 *   v_scales           [n_blocks][n_kv_heads][block_size][head_dim / 32]
 *                      fp16 bits, one per 32 dims
 *
 * where the dims are those of the rotated row y = H v (H the Walsh-Hadamard
 * matrix of order head_dim, Sylvester order, entries +-1), so a cell costs
 * 2 * n_kv_heads * (head_dim + head_dim / 32) + n_kv_heads * head_dim * 18 /
 * 32 bytes: 816 at 2 KV heads of 256 dims ([k8v4 PR], "What").
 *
 * Cell p of sequence b is block block_table[b * max_blocks_per_seq +
 * p / block_size], slot p % block_size; its row of KV head h starts at
 * element ((block * n_kv_heads + h) * block_size + slot) * head_dim.
 *
 * Limits: head_dim in {64, 128, 256}; block_size a power of two in
 * [16, 1024]; all four pointers 256-byte aligned (torch allocations are);
 * n_blocks * n_kv_heads * block_size < 2^31.
 */
typedef struct kvq_cache {
    int32_t fmt;        /* kvq_format */
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t n_blocks;
    int32_t reserved;   /* must be 0 */
    void *k_data;
    void *v_data;
    void *k_scales;
    void *v_scales;
} kvq_cache;

/*
 * Bytes one physical block occupies in the pool: K and V codes plus, for
 * KVQ_Q8, their scales (2 bytes per 64 dims).  Per element that is 2 bytes
 * (F16) or 1 + 2/64 bytes (Q8) -- the 6.0 GiB and 3.1 GiB of a 262144-cell
 * cache in [kv-q8 PR], "Summary".  KVQ_K8V4: 1 + 2/64 bytes per K element
 * and 18/32 per V element.  Returns 0 for an invalid geometry.
 */
size_t kvq_block_bytes(int fmt, int n_kv_heads, int head_dim, int block_size);

/*
 * Quantize-on-write of n_tok new cells ([kv-q8 PR], "What changed";
 * [k8v4 PR], "How": one call serves the decode step (n_tok = number of
 * sequences), a verify window and a prompt chunk).
 *
 *   k, v        device fp32 [n_tok][n_kv_heads][head_dim], 16-byte aligned
 *   tok_seq     device int32 [n_tok]: sequence of each new cell
 *   tok_pos     device int32 [n_tok]: its position (cell index) in that
 *               sequence
 *   block_table device int32 [n_seq][max_blocks_per_seq]
 *   n_seq       host int: rows of block_table (bounds tok_seq)
 *
 * KVQ_F16 stores fp16_rne(x).  KVQ_Q8 stores, per row and per group of 64
 * dims, s = fp16_rne(max|x| / 127) and codes clamp(rint(x / float(s)), -127,
 * 127): both divisions are IEEE fp32 divisions, rint rounds half to even; a
 * group whose scale is 0 gets zero codes.  The result is bit-identical to
 * that definition.  KVQ_K8V4 writes K that way; V is first rotated, y = H v,
 * in fp32 by butterflies (stages h = 1, 2, ..., head_dim / 2; in each, dims
 * j and j + h, bit h of j clear, become their sum and difference), then
 * each block of 32 dims of y gets d = fp16_rne(m / -8), m the block's
 * element of largest magnitude (the first one on ties), and codes
 * clamp(rint(y / float(d)), -8, 7) + 8 (8 when d is 0), both divisions
 * IEEE fp32.  A cell written twice holds the last write; two tokens of
 * one call must not name the same cell.  n_tok == 0 is a no-op returning
 * KVQ_OK.
 */
kvq_status kvq_append(const kvq_cache *cache, const float *k, const float *v, int n_tok,
                      const int32_t *tok_seq, const int32_t *tok_pos,
                      const int32_t *block_table, int n_seq, int max_blocks_per_seq,
                      void *stream);

/*
 * Workspace bytes kvq_decode_attn needs for these sizes on the current
 * device (the split plan depends on its SM count).  Returns 0 for invalid
 * arguments.
 */
size_t kvq_decode_workspace_bytes(const kvq_cache *cache, int n_seq, int W, int n_q,
                                  int max_ctx);

/*
 * Decode attention of W query tokens per sequence against the cache
 * ([kv-q8 PR], "What changed" and "Extra Notes": the split-K partial kernel
 * k_attn_part and its combine).
 *
 *   q           device fp32 [n_seq][W][n_q][head_dim], 16-byte aligned
 *   ctx_lens    device int32 [n_seq]: cells in each sequence, the W query
 *               tokens' own cells included (they are appended first)
 *   max_ctx     host int: an upper bound of ctx_lens, used to plan splits
 *   block_table device int32 [n_seq][max_blocks_per_seq]
 *   sm_scale    softmax scale (usually 1/sqrt(head_dim))
 *   out         device fp32 [n_seq][W][n_q][head_dim], 16-byte aligned
 *   workspace   device scratch of at least kvq_decode_workspace_bytes(),
 *               256-byte aligned; no initial contents are needed.  It
 *               holds the split-K partials between the partial kernel and
 *               the combine kernel of one call, so calls sharing a
 *               workspace must be ordered (same stream, or events).
 *
 * Query head h reads KV head h / (n_q / n_kv_heads); n_q must be a
 * multiple of n_kv_heads.  Query token w of sequence b is the cell
 * ctx_lens[b] - W + w and attends to cells [0, ctx_lens[b] - W + w]
 * (causal inside the window).  out = softmax(sm_scale * q . K^T) V over the
 * dequantized cache, computed in fp32; a query with no visible cell gets 0.
 * For KVQ_K8V4 the dequantized V is the rotated one, (code - 8) * d, and
 * the result is rotated back, out = H o / head_dim.
 * W in [1, 16], n_q / n_kv_heads * W <= 32.
 */
kvq_status kvq_decode_attn(const kvq_cache *cache, const float *q, int n_seq, int W, int n_q,
                           const int32_t *ctx_lens, int max_ctx, const int32_t *block_table,
                           int max_blocks_per_seq, float sm_scale, float *out,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * kvq_decode_attn with the failure path of its copy waits exercised, for
 * tests of that path only.  Every wait of the tensor-core decode for a
 * copy into shared memory is bounded; a wait that runs out marks the
 * split's partial as lost, the combine writes NaN for the affected output
 * rows, and the kernel still waits (bounded) for its own copies before it
 * exits, so the context stays usable.  This call adds extra_tx_bytes
 * (a multiple of 16 in [16, 4096]) to the byte count every copy stage
 * expects, bytes no copy ever delivers, and bounds each wait by
 * wait_limit polls (1 .. 2^25; kvq_decode_attn uses 2^25): every wait runs
 * out, and a correct failure path returns KVQ_OK with NaN in every output
 * row of a sequence with cells.  No fault, trap or unbounded wait is
 * involved.  Other arguments, checks and errors as kvq_decode_attn; shapes
 * that the tensor-core kernel does not serve return KVQ_ERR_UNSUPPORTED.
 */
kvq_status kvq_decode_attn_lost_wait_test(const kvq_cache *cache, const float *q, int n_seq,
                                          int W, int n_q, const int32_t *ctx_lens, int max_ctx,
                                          const int32_t *block_table, int max_blocks_per_seq,
                                          float sm_scale, float *out, void *workspace,
                                          size_t workspace_bytes, uint32_t wait_limit,
                                          uint32_t extra_tx_bytes, void *stream);

/*
 * FP16 compaction of cells [0, n_cells) of one sequence ([kv-q8 PR],
 * "Extra Notes": k_kv_f16 compacts [kvh][ctx][HD] into [kvh][P][HD]
 * halves; on the FP16 cache it is a pure copy).
 *
 *   block_table_row device int32 [ceil(n_cells / block_size)]: the
 *                   sequence's row of the block table
 *   out_k, out_v    device fp16 [n_kv_heads][n_cells][head_dim], 16-byte
 *                   aligned
 *
 * KVQ_F16 copies the stored bits; KVQ_Q8 writes fp16_rne(code * scale)
 * (the product is exact in fp32).  KVQ_K8V4 writes K that way and V as
 * fp16_rne(w / head_dim), w the fp32 butterflies of kvq_append applied to
 * the row of (code - 8) * d (the inverse rotation).  n_cells == 0 is a
 * no-op.
 */
kvq_status kvq_compact_f16(const kvq_cache *cache, const int32_t *block_table_row, int n_cells,
                           void *out_k, void *out_v, void *stream);

/*
 * Attention of a prompt chunk over the FP16 staging ([kv-q8 PR], "Extra
 * Notes": the prompt chunk's Q K^T and P V products read the contiguous
 * [kvh][P][HD] fp16 halves that k_kv_f16 writes).
 *
 *   k16, v16   device fp16 [n_kv_heads][P][head_dim], 16-byte aligned: the
 *              sequence's P cells as kvq_compact_f16 writes them
 *   q          device fp32 [T][n_q][head_dim], 16-byte aligned: the chunk's
 *              T query tokens, which are the sequence's last T cells
 *   out        device fp32 [T][n_q][head_dim], 16-byte aligned
 *
 * Token t attends to cells [0, P - T + t] (causal); query head h reads KV
 * head h / (n_q / n_kv_heads).  out = softmax(sm_scale * q . K^T) V with
 * fp32 accumulation (q enters the tensor cores as an fp16 hi + lo pair, the
 * softmax weights as one fp16 value).  head_dim in {64, 128, 256}; 1 <= T <= P;
 * n_q a multiple of n_kv_heads; n_kv_heads * P < 2^31.  Invalid arguments
 * return KVQ_ERR_ARG / KVQ_ERR_UNSUPPORTED before any launch.  Asynchronous
 * on `stream`; the library allocates nothing.
 */
kvq_status kvq_chunk_attn(const void *k16, const void *v16, int n_kv_heads, int P, int head_dim,
                          const float *q, int T, int n_q, float sm_scale, float *out,
                          void *stream);

/*
 * kvq_chunk_attn with the failure path of its waits exercised, for tests of
 * that path only.  Every mbarrier wait of the chunk kernel is bounded; a
 * wait that runs out turns the CTA's rows into NaN (through the merge too,
 * when a short chunk's key tiles are split over a cluster of CTAs), and
 * each role still waits (bounded) for its own copies and MMAs before the
 * CTA exits, so the context stays usable.  This call adds extra_tx_bytes
 * (a multiple of 16 in [16, 4096]) to the byte count every K and V stage
 * expects, bytes no copy ever delivers, and bounds each wait by wait_limit
 * polls (1 .. 2^25; kvq_chunk_attn uses 2^25): every wait runs out, and a
 * correct failure path returns KVQ_OK with NaN in every output row.  No
 * fault, trap or unbounded wait is involved.  Other arguments, checks and
 * errors as kvq_chunk_attn.
 */
kvq_status kvq_chunk_attn_lost_wait_test(const void *k16, const void *v16, int n_kv_heads, int P,
                                         int head_dim, const float *q, int T, int n_q,
                                         float sm_scale, float *out, uint32_t wait_limit,
                                         uint32_t extra_tx_bytes, void *stream);

/*
 * Persistence of one sequence: cells [0, n_cells) gathered out of the pool
 * into token-major runs, and scattered back into a pool (Path F format v3:
 * persist per-head INT8 KV scales for INT8 + persistent KV interop,
 * "Scope": a saved turn is its used cells' K/V bytes followed by their
 * scales; "Why": int8 bytes without the scales would hydrate to garbage).
 *
 *   block_table_row  device int32 [ceil(n_cells / block_size)]: the
 *                    sequence's row of the block table
 *   codes_k, codes_v device [n_cells][n_kv_heads][head_dim] elements of the
 *                    pool's format (fp16 or int8), 16-byte aligned; K8V4's
 *                    codes_v is [n_cells][n_kv_heads][head_dim / 2] bytes
 *   scales_k, scales_v
 *                    device fp16 [n_cells][n_kv_heads][head_dim / 64], 16-byte
 *                    aligned; required
 *                    for KVQ_Q8 (KVQ_ERR_ARG without them), ignored for
 *                    KVQ_F16; K8V4 requires both, scales_v being
 *                    [n_cells][n_kv_heads][head_dim / 32]
 *
 * Both copy bits unchanged: a gather followed by a scatter into any pool
 * of the same format and geometry, under any block table, restores the
 * cells exactly.  Cells whose block id is out of range are skipped.
 * n_cells == 0 is a no-op.  Asynchronous on `stream`.
 */
kvq_status kvq_gather_cells(const kvq_cache *cache, const int32_t *block_table_row, int n_cells,
                            void *codes_k, void *codes_v, void *scales_k, void *scales_v,
                            void *stream);
kvq_status kvq_scatter_cells(const kvq_cache *cache, const int32_t *block_table_row, int n_cells,
                             const void *codes_k, const void *codes_v, const void *scales_k,
                             const void *scales_v, void *stream);

/*
 * Block streaming with a resident window ([k8v4 PR], "What" and "How": the
 * cache's authoritative copy lives in pinned host memory and a window of
 * N cells' worth of device blocks holds what the GPU reads; a block moves
 * as its list of byte runs, so every format streams the same way; "Tests":
 * attention over the streamed state is bitwise equal to attention over a
 * fully resident pool).
 *
 * The host copy is a kvq_cache whose four arrays are pinned host memory
 * the device can address (cudaHostAlloc'd or registered, mapped; on a
 * Grace-Blackwell node the kernels reach it over NVLink-C2C), n_blocks of
 * them; the window is an ordinary device kvq_cache of n_slots blocks with
 * the same format and geometry.  Appends go to both (the host copy under
 * the sequences' block table, the window under the slot table, where
 * non-resident blocks are -1 and therefore skipped); attention and
 * compaction read the window under the slot table.  One step:
 *
 *   kvq_append(host copy, block_table)        authoritative write
 *   kvq_stream_plan(..., block_table, ctx)    slots, fetch list (host)
 *   kvq_stream_fetch(host copy, window, list) missing blocks -> slots
 *   kvq_append(window, slot_table)            resident blocks' new cells
 *   kvq_decode_attn(window, slot_table)
 */

/*
 * Residency plan for one call, host only (no device access, nothing
 * launched).  The residency state is three caller-owned host arrays and a
 * counter, initialised by the caller to -1 / -1 / 0 / 0:
 *
 *   slot_of_block [n_host_blocks]  int32: window slot of a host block, -1
 *   block_of_slot [n_slots]        int32: host block in a slot, -1 if free
 *   last_use      [n_slots]        int64: the counter value of the slot's
 *                                  last plan
 *   clock                          int64: advanced by one per plan
 *
 * Inputs (host int32): block_table [n_seq][max_blocks_per_seq] of host
 * block ids, ctx_lens [n_seq] (cells each sequence's call reads, its new
 * cells included), block_size.  The call reads blocks [0, ceil(ctx_lens[b]
 * / block_size)) of each row; ids outside [0, n_host_blocks) are ignored.
 * Every distinct block read gets a slot: a resident one keeps its slot (a
 * hit); the others take, in order of first use, free slots in index
 * order, then the slots this call does not read, least recently used first
 * (ties: lower index).  Outputs (host): slot_table [n_seq][max_blocks_per_seq]
 * (the slot of each entry's block, -1 where it is not resident),
 * fetch_src / fetch_dst [capacity n_slots] the (host block, slot) pairs
 * to fetch, *n_fetch their count, *n_hits (may be NULL) the hits.  A call
 * that reads more distinct blocks than n_slots returns KVQ_ERR_UNSUPPORTED
 * and changes nothing; invalid sizes or NULL arrays return KVQ_ERR_ARG.
 * The function uses temporary host memory and keeps no state of its own.
 */
kvq_status kvq_stream_plan(int n_host_blocks, int n_slots, int32_t *slot_of_block,
                           int32_t *block_of_slot, int64_t *last_use, int64_t *clock,
                           const int32_t *block_table, int n_seq, int max_blocks_per_seq,
                           const int32_t *ctx_lens, int block_size, int32_t *slot_table,
                           int32_t *fetch_src, int32_t *fetch_dst, int *n_fetch, int *n_hits);

/*
 * Copy n_fetch blocks from the host copy into window slots: block
 * fetch_src[i] of every run of host_copy goes to block fetch_dst[i] of the
 * same run of window, bits unchanged (two runs for KVQ_F16, four
 * otherwise).  One kernel reads the host memory directly (16-byte loads,
 * several in flight per thread) and writes the window; no copy engine is
 * involved.  fetch_src / fetch_dst: int32 [n_fetch] that the device can
 * read (device memory or mapped pinned host memory, e.g. the plan's
 * outputs in pinned memory).  Both caches must pass the kvq_append checks
 * and agree in format, n_kv_heads, head_dim and block_size (else
 * KVQ_ERR_ARG); every array of the host copy must be device-addressable
 * at its own address (the runtime's pointer attributes give it that device
 * address: pinned memory under unified addressing, device or managed
 * memory), so that kvq_append can write it too, else KVQ_ERR_ARG -- checked
 * even when n_fetch is 0, so a call with n_fetch 0 validates a host copy
 * before anything writes to it.  Ids out of range skip their fetch.  Two
 * fetches must not name the same slot.  Asynchronous on `stream`.
 */
kvq_status kvq_stream_fetch(const kvq_cache *host_copy, const kvq_cache *window,
                            const int32_t *fetch_src, const int32_t *fetch_dst, int n_fetch,
                            void *stream);

/*
 * Bytes of device scratch that kvq_decode_attn_static keeps in the library
 * (one array per device that loads the library, held until the process
 * exits).
 */
#define KVQ_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * kvq_decode_attn without a workspace argument, for callers that cannot
 * allocate device memory: code running during CUDA graph capture (where
 * cudaMalloc is not allowed), plugins inside a framework whose allocator
 * owns the device memory, real-time loops whose memory is fixed at
 * start-up.  The paper has no counterpart to this call; it exists for
 * such callers only.
 *
 * Arguments, results and errors are those of kvq_decode_attn.  The scratch
 * is a file-scope device array of KVQ_STATIC_SCRATCH_BYTES inside the
 * library; when the split plan kvq_decode_workspace_bytes describes needs
 * more, the context is cut into fewer splits until it fits, and a request
 * that does not fit even with one split per (sequence, KV head) returns
 * KVQ_ERR_WORKSPACE and launches nothing.  The first call on a device
 * looks up the array's address and caches it for that device's context
 * (looked up again after the context changes, e.g. after cudaDeviceReset):
 * make that first call before any stream capture.
 * Every call uses the same array, so calls whose kernels may overlap on
 * the GPU (unordered streams) race on it; order them.  The array needs no
 * clearing between calls.
 */
kvq_status kvq_decode_attn_static(const kvq_cache *cache, const float *q, int n_seq, int W,
                                  int n_q, const int32_t *ctx_lens, int max_ctx,
                                  const int32_t *block_table, int max_blocks_per_seq,
                                  float sm_scale, float *out, void *stream);

/* Static, human-readable name of a status code. */
const char *kvq_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */

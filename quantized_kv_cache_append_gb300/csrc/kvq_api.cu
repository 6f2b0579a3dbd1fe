// kvq_api.cu -- the C ABI (include/kvq.h): host-side validation, split
// planning and launches.  Nothing here reads device memory or synchronizes.
//
// Error rules follow the pages' "refuse rather than silently skip":
// #711 kv: --kv k8v4 streams with --kv-resident, "How" (a writer that tested
// one pointer and silently skipped the other) and "Tests" (the negative
// control that catches it); Path F format v3: persist per-head INT8 KV
// scales, "Why" and "Scope" (int8 bytes without their scales are refused).
// So a missing scale pointer, like every other invalid argument, is an
// error returned before any launch.
#include <math.h>
#include <stdint.h>

#include "kvq_internal.cuh"

#define KVQ_API extern "C" __attribute__((visibility("default")))

namespace kvq {
namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int log2_exact(int v) {
  int l = 0;
  while ((1 << l) < v) ++l;
  return (1 << l) == v ? l : -1;
}

// Geometry checks shared by every call.
kvq_status check_cache(const kvq_cache* c) {
  if (c == nullptr) return KVQ_ERR_ARG;
  if (c->fmt != KVQ_F16 && c->fmt != KVQ_Q8 && c->fmt != KVQ_K8V4) return KVQ_ERR_ARG;
  if (c->reserved != 0) return KVQ_ERR_ARG;
  if (c->n_kv_heads <= 0 || c->n_blocks <= 0) return KVQ_ERR_ARG;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return KVQ_ERR_ARG;
  if (c->block_size < 16 || c->block_size > 1024 || log2_exact(c->block_size) < 0)
    return KVQ_ERR_ARG;
  if ((long long)c->n_blocks * c->n_kv_heads * c->block_size >= (1LL << 31)) return KVQ_ERR_ARG;
  if (c->k_data == nullptr || c->v_data == nullptr) return KVQ_ERR_ARG;
  if (!aligned(c->k_data, 256) || !aligned(c->v_data, 256)) return KVQ_ERR_ARG;
  if (c->fmt != KVQ_F16) {
    // int8 (or 4-bit) codes without their scales are refused, never half-written.
    if (c->k_scales == nullptr || c->v_scales == nullptr) return KVQ_ERR_ARG;
    if (!aligned(c->k_scales, 256) || !aligned(c->v_scales, 256)) return KVQ_ERR_ARG;
  }
  return KVQ_OK;
}

Pool make_pool(const kvq_cache* c) {
  Pool p;
  p.k = c->k_data;
  p.v = c->v_data;
  p.ks = static_cast<const __half*>(c->k_scales);
  p.vs = static_cast<const __half*>(c->v_scales);
  p.n_kv = c->n_kv_heads;
  p.bs_log2 = log2_exact(c->block_size);
  p.n_blocks = c->n_blocks;
  return p;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Split plan: one wave of partial CTAs (as many as are resident per SM, on
// every SM; four times that for batches, whose ragged lengths need short
// splits to fill the tail of the launch) over all (sequence, KV head, row
// tile) items, each split a whole number of cell tiles.  A verify window
// wider than one CTA's rows is cut into row tiles of mma_rows_per_cta rows.
// With max_bytes set, the split count is lowered until the workspace fits
// (false if even one split per pair does not).  use_mma is 0 when the
// kernel's one-time setup failed.
bool plan_decode(const kvq_cache* c, int n_seq, int W, int n_q, int max_ctx, DecodePlan* p,
                 size_t max_bytes = SIZE_MAX) {
  const int G = n_q / c->n_kv_heads;
  p->rows = G * W;
  const int cta_rows = mma_rows_per_cta(c->head_dim);
  p->rt_rows = p->rows < cta_rows ? p->rows : cta_rows;
  p->n_rt = (p->rows + p->rt_rows - 1) / p->rt_rows;
  int per_sm = mma_ctas_per_sm(c->fmt, c->head_dim, p->rt_rows);
  p->use_mma = per_sm > 0;
  if (!p->use_mma) per_sm = 1;   // still a plan (and a workspace size); the launch is refused
  const int tile = mma_cell_tile();
  const long long units = (long long)n_seq * c->n_kv_heads * p->n_rt;
  const int tiles = (max_ctx + tile - 1) / tile;
  int sms = sm_count();
  if (sms <= 0) sms = 148;
  const long long capacity = (long long)per_sm * sms;
  const long long target = capacity * (n_seq > 1 ? 4 : 1);
  long long ns = target / units;
  if (ns < 1) ns = 1;
  if (ns > tiles) ns = tiles;
  for (;;) {
    const int split_tiles = (int)((tiles + ns - 1) / ns);
    p->split_cells = split_tiles * tile;
    p->nsplit = (max_ctx + p->split_cells - 1) / p->split_cells;
    const size_t parts = (size_t)n_seq * c->n_kv_heads * p->nsplit * p->rows;
    p->off_o = 0;
    p->off_ml = round_up(parts * c->head_dim * sizeof(float), 256);
    p->bytes = p->off_ml + round_up(parts * 2 * sizeof(float), 256);
    if (p->bytes <= max_bytes) return true;
    if (p->nsplit <= 1) return false;
    // shrink in proportion, at least by one split
    long long next = (long long)((double)p->nsplit * (double)max_bytes / (double)p->bytes);
    ns = next < p->nsplit - 1 ? next : p->nsplit - 1;
    if (ns < 1) ns = 1;
  }
}

kvq_status check_decode_shape(const kvq_cache* c, int n_seq, int W, int n_q, int max_ctx,
                              int max_blocks) {
  if (n_seq <= 0 || n_q <= 0 || max_ctx <= 0 || max_blocks <= 0) return KVQ_ERR_ARG;
  if (W < 1 || W > 16) return KVQ_ERR_ARG;
  if (n_q % c->n_kv_heads != 0) return KVQ_ERR_ARG;
  if (max_ctx < W) return KVQ_ERR_ARG;
  if ((long long)max_ctx > (long long)max_blocks * c->block_size) return KVQ_ERR_ARG;
  if (n_seq > 65535 || c->n_kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
  const int rows = (n_q / c->n_kv_heads) * W;
  if (!mma_decode_supported(c->fmt, c->head_dim, rows)) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

}  // namespace
}  // namespace kvq

using namespace kvq;

KVQ_API size_t kvq_block_bytes(int fmt, int n_kv_heads, int head_dim, int block_size) {
  if (n_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return 0;
  const size_t elems = (size_t)n_kv_heads * head_dim * block_size;  // per K (or V)
  if (fmt == KVQ_F16) return 2 * elems * 2;
  if (fmt == KVQ_Q8) {
    if (head_dim % KVQ_GROUP != 0) return 0;
    return 2 * (elems + (elems / KVQ_GROUP) * 2);
  }
  if (fmt == KVQ_K8V4) {
    if (head_dim % KVQ_GROUP != 0) return 0;
    return elems + (elems / KVQ_GROUP) * 2 + elems / 2 + (elems / KVQ_Q4_BLOCK) * 2;
  }
  return 0;
}

KVQ_API kvq_status kvq_append(const kvq_cache* cache, const float* k, const float* v, int n_tok,
                              const int32_t* tok_seq, const int32_t* tok_pos,
                              const int32_t* block_table, int n_seq, int max_blocks_per_seq,
                              void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_tok < 0) return KVQ_ERR_ARG;
  if (n_tok == 0) return KVQ_OK;
  if (k == nullptr || v == nullptr || tok_seq == nullptr || tok_pos == nullptr ||
      block_table == nullptr)
    return KVQ_ERR_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(tok_seq, 4) || !aligned(tok_pos, 4) ||
      !aligned(block_table, 4))
    return KVQ_ERR_ARG;
  if (n_seq <= 0 || max_blocks_per_seq <= 0) return KVQ_ERR_ARG;
  if ((long long)n_tok * cache->n_kv_heads * 2 >= (1LL << 36)) return KVQ_ERR_UNSUPPORTED;
  AppendArgs a;
  a.k_dst = cache->k_data;
  a.v_dst = cache->v_data;
  a.ks_dst = static_cast<__half*>(cache->k_scales);
  a.vs_dst = static_cast<__half*>(cache->v_scales);
  a.k = k;
  a.v = v;
  a.tok_seq = tok_seq;
  a.tok_pos = tok_pos;
  a.block_table = block_table;
  a.n_tok = n_tok;
  a.n_kv = cache->n_kv_heads;
  a.bs_log2 = log2_exact(cache->block_size);
  a.n_blocks = cache->n_blocks;
  a.n_seq = n_seq;
  a.max_blocks = max_blocks_per_seq;
  const cudaError_t e =
      launch_append(cache->fmt, cache->head_dim, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

KVQ_API size_t kvq_decode_workspace_bytes(const kvq_cache* cache, int n_seq, int W, int n_q,
                                          int max_ctx) {
  if (check_cache(cache) != KVQ_OK) return 0;
  const int max_blocks = (max_ctx + cache->block_size - 1) / cache->block_size;
  if (check_decode_shape(cache, n_seq, W, n_q, max_ctx, max_blocks > 0 ? max_blocks : 1) !=
      KVQ_OK)
    return 0;
  DecodePlan p;
  if (!plan_decode(cache, n_seq, W, n_q, max_ctx, &p)) return 0;
  return p.bytes;
}

namespace kvq {
namespace {

// Validation, plan and launch of one decode call.  fit_plan: lower the split
// count until the plan fits workspace_bytes (the static-scratch entry
// point); otherwise the full plan must fit.
kvq_status decode_impl(const kvq_cache* cache, const float* q, int n_seq, int W, int n_q,
                       const int32_t* ctx_lens, int max_ctx, const int32_t* block_table,
                       int max_blocks_per_seq, float sm_scale, float* out, void* workspace,
                       size_t workspace_bytes, void* stream, bool fit_plan,
                       uint32_t wait_limit = kDefaultWaitLimit, uint32_t extra_tx = 0) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  st = check_decode_shape(cache, n_seq, W, n_q, max_ctx, max_blocks_per_seq);
  if (st != KVQ_OK) return st;
  if (q == nullptr || out == nullptr || ctx_lens == nullptr || block_table == nullptr)
    return KVQ_ERR_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(ctx_lens, 4) || !aligned(block_table, 4))
    return KVQ_ERR_ARG;
  if (!(sm_scale == sm_scale) || isinf(sm_scale)) return KVQ_ERR_ARG;
  if (workspace == nullptr || !aligned(workspace, 256)) return KVQ_ERR_WORKSPACE;
  DecodePlan plan;
  if (!plan_decode(cache, n_seq, W, n_q, max_ctx, &plan, fit_plan ? workspace_bytes : SIZE_MAX))
    return fit_plan ? KVQ_ERR_WORKSPACE : KVQ_ERR_ARG;
  if (workspace_bytes < plan.bytes) return KVQ_ERR_WORKSPACE;
  if (!plan.use_mma) return KVQ_ERR_CUDA;   // the kernels' one-time setup failed
  DecodeArgs a;
  a.pool = make_pool(cache);
  a.q = q;
  a.out = out;
  a.ctx_lens = ctx_lens;
  a.block_table = block_table;
  a.ws_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.off_o);
  a.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.off_ml);
  a.n_seq = n_seq;
  a.W = W;
  a.n_q = n_q;
  a.G = n_q / cache->n_kv_heads;
  a.g_magic = (0x100000000ull + (unsigned long long)a.G - 1) / (unsigned long long)a.G;
  a.div_nkv = make_fastdiv((unsigned)cache->n_kv_heads);
  a.div_nrt = make_fastdiv((unsigned)plan.n_rt);
  a.div_split = make_fastdiv((unsigned)plan.split_cells);
  a.R = plan.rows;
  a.RT = plan.rt_rows;
  a.n_rt = plan.n_rt;
  a.max_blocks = max_blocks_per_seq;
  a.split_cells = plan.split_cells;
  a.nsplit = plan.nsplit;
  a.qscale = sm_scale * 1.4426950408889634f;  // log2(e)
  a.wait_limit = wait_limit;
  a.extra_tx = extra_tx;
  const cudaError_t e = launch_decode_mma_partial(cache->fmt, cache->head_dim, plan, a,
                                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace
}  // namespace kvq

KVQ_API kvq_status kvq_decode_attn(const kvq_cache* cache, const float* q, int n_seq, int W,
                                   int n_q, const int32_t* ctx_lens, int max_ctx,
                                   const int32_t* block_table, int max_blocks_per_seq,
                                   float sm_scale, float* out, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return kvq::decode_impl(cache, q, n_seq, W, n_q, ctx_lens, max_ctx, block_table,
                          max_blocks_per_seq, sm_scale, out, workspace, workspace_bytes, stream,
                          false);
}

KVQ_API kvq_status kvq_decode_attn_lost_wait_test(const kvq_cache* cache, const float* q, int n_seq,
                                                  int W, int n_q, const int32_t* ctx_lens,
                                                  int max_ctx, const int32_t* block_table,
                                                  int max_blocks_per_seq, float sm_scale, float* out,
                                                  void* workspace, size_t workspace_bytes,
                                                  uint32_t wait_limit, uint32_t extra_tx_bytes,
                                                  void* stream) {
  if (wait_limit == 0 || wait_limit > kDefaultWaitLimit) return KVQ_ERR_ARG;
  if (extra_tx_bytes == 0 || extra_tx_bytes > 4096 || extra_tx_bytes % 16 != 0) return KVQ_ERR_ARG;
  return kvq::decode_impl(cache, q, n_seq, W, n_q, ctx_lens, max_ctx, block_table,
                          max_blocks_per_seq, sm_scale, out, workspace, workspace_bytes, stream,
                          false, wait_limit, extra_tx_bytes);
}

KVQ_API kvq_status kvq_compact_f16(const kvq_cache* cache, const int32_t* block_table_row,
                                   int n_cells, void* out_k, void* out_v, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_cells < 0) return KVQ_ERR_ARG;
  if (n_cells == 0) return KVQ_OK;
  if (block_table_row == nullptr || out_k == nullptr || out_v == nullptr) return KVQ_ERR_ARG;
  if (!aligned(block_table_row, 4) || !aligned(out_k, 16) || !aligned(out_v, 16))
    return KVQ_ERR_ARG;
  CompactArgs a;
  a.pool = make_pool(cache);
  a.block_row = block_table_row;
  a.n_cells = n_cells;
  a.out_k = static_cast<__half*>(out_k);
  a.out_v = static_cast<__half*>(out_v);
  const cudaError_t e =
      launch_compact(cache->fmt, cache->head_dim, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

namespace kvq {
namespace {

kvq_status persist_impl(const kvq_cache* cache, const int32_t* block_table_row, int n_cells,
                        const void* codes_k, const void* codes_v, const void* scales_k,
                        const void* scales_v, bool gather, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_cells < 0) return KVQ_ERR_ARG;
  if (n_cells == 0) return KVQ_OK;
  if (block_table_row == nullptr || codes_k == nullptr || codes_v == nullptr) return KVQ_ERR_ARG;
  // int8 (and 4-bit) codes never move without their scales
  if (cache->fmt != KVQ_F16 && (scales_k == nullptr || scales_v == nullptr)) return KVQ_ERR_ARG;
  if (!aligned(block_table_row, 4) || !aligned(codes_k, 16) || !aligned(codes_v, 16) ||
      !aligned(scales_k, 16) || !aligned(scales_v, 16))
    return KVQ_ERR_ARG;
  if ((long long)n_cells * cache->n_kv_heads >= (1LL << 31)) return KVQ_ERR_UNSUPPORTED;
  PersistArgs a;
  a.pool = make_pool(cache);
  a.pool_k = cache->k_data;
  a.pool_v = cache->v_data;
  a.pool_ks = static_cast<__half*>(cache->k_scales);
  a.pool_vs = static_cast<__half*>(cache->v_scales);
  a.block_row = block_table_row;
  a.n_cells = n_cells;
  a.codes_k = const_cast<void*>(codes_k);
  a.codes_v = const_cast<void*>(codes_v);
  a.scales_k = static_cast<__half*>(const_cast<void*>(scales_k));
  a.scales_v = static_cast<__half*>(const_cast<void*>(scales_v));
  const cudaError_t e =
      launch_persist(cache->fmt, cache->head_dim, gather, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace
}  // namespace kvq

KVQ_API kvq_status kvq_gather_cells(const kvq_cache* cache, const int32_t* block_table_row,
                                    int n_cells, void* codes_k, void* codes_v, void* scales_k,
                                    void* scales_v, void* stream) {
  return kvq::persist_impl(cache, block_table_row, n_cells, codes_k, codes_v, scales_k, scales_v,
                           true, stream);
}

KVQ_API kvq_status kvq_scatter_cells(const kvq_cache* cache, const int32_t* block_table_row,
                                     int n_cells, const void* codes_k, const void* codes_v,
                                     const void* scales_k, const void* scales_v, void* stream) {
  return kvq::persist_impl(cache, block_table_row, n_cells, codes_k, codes_v, scales_k, scales_v,
                           false, stream);
}

namespace kvq {
namespace {
kvq_status chunk_impl(const void* k16, const void* v16, int n_kv_heads, int P, int head_dim,
                      const float* q, int T, int n_q, float sm_scale, float* out, void* stream,
                      uint32_t wait_limit = kDefaultWaitLimit, uint32_t extra_tx = 0) {
  if (k16 == nullptr || v16 == nullptr || q == nullptr || out == nullptr) return KVQ_ERR_ARG;
  if (!aligned(k16, 16) || !aligned(v16, 16) || !aligned(q, 16) || !aligned(out, 16))
    return KVQ_ERR_ARG;
  if (n_kv_heads <= 0 || P <= 0 || T <= 0 || T > P || n_q <= 0 || n_q % n_kv_heads != 0)
    return KVQ_ERR_ARG;
  if (!(sm_scale == sm_scale) || isinf(sm_scale)) return KVQ_ERR_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  if ((long long)n_kv_heads * P >= (1LL << 31) || (long long)T * n_q >= (1LL << 31) ||
      n_kv_heads > 65535)
    return KVQ_ERR_UNSUPPORTED;
  ChunkArgs a;
  a.k16 = static_cast<const __half*>(k16);
  a.v16 = static_cast<const __half*>(v16);
  a.q = q;
  a.out = out;
  a.n_kv = n_kv_heads;
  a.P = P;
  a.T = T;
  a.n_q = n_q;
  a.G = n_q / n_kv_heads;
  a.qscale = sm_scale * 1.4426950408889634f;  // log2(e)
  a.wait_limit = wait_limit;
  a.extra_tx = extra_tx;
  const cudaError_t e = launch_chunk_attn(head_dim, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
}  // namespace
}  // namespace kvq

KVQ_API kvq_status kvq_chunk_attn(const void* k16, const void* v16, int n_kv_heads, int P,
                                  int head_dim, const float* q, int T, int n_q, float sm_scale,
                                  float* out, void* stream) {
  return kvq::chunk_impl(k16, v16, n_kv_heads, P, head_dim, q, T, n_q, sm_scale, out, stream);
}

KVQ_API kvq_status kvq_chunk_attn_lost_wait_test(const void* k16, const void* v16, int n_kv_heads,
                                                 int P, int head_dim, const float* q, int T, int n_q,
                                                 float sm_scale, float* out, uint32_t wait_limit,
                                                 uint32_t extra_tx_bytes, void* stream) {
  if (wait_limit == 0 || wait_limit > kDefaultWaitLimit) return KVQ_ERR_ARG;
  if (extra_tx_bytes == 0 || extra_tx_bytes > 4096 || extra_tx_bytes % 16 != 0) return KVQ_ERR_ARG;
  return kvq::chunk_impl(k16, v16, n_kv_heads, P, head_dim, q, T, n_q, sm_scale, out, stream,
                         wait_limit, extra_tx_bytes);
}

KVQ_API kvq_status kvq_stream_plan(int n_host_blocks, int n_slots, int32_t* slot_of_block,
                                   int32_t* block_of_slot, int64_t* last_use, int64_t* clock,
                                   const int32_t* block_table, int n_seq, int max_blocks_per_seq,
                                   const int32_t* ctx_lens, int block_size, int32_t* slot_table,
                                   int32_t* fetch_src, int32_t* fetch_dst, int* n_fetch,
                                   int* n_hits) {
  if (n_host_blocks <= 0 || n_slots <= 0 || n_seq < 0 || max_blocks_per_seq <= 0 || block_size <= 0)
    return KVQ_ERR_ARG;
  if (slot_of_block == nullptr || block_of_slot == nullptr || last_use == nullptr ||
      clock == nullptr || fetch_src == nullptr || fetch_dst == nullptr || n_fetch == nullptr)
    return KVQ_ERR_ARG;
  if (n_seq > 0 && (block_table == nullptr || ctx_lens == nullptr || slot_table == nullptr))
    return KVQ_ERR_ARG;
  return kvq::stream_plan(n_host_blocks, n_slots, slot_of_block, block_of_slot, last_use, clock,
                          block_table, n_seq, max_blocks_per_seq, ctx_lens, block_size, slot_table,
                          fetch_src, fetch_dst, n_fetch, n_hits);
}

KVQ_API kvq_status kvq_stream_fetch(const kvq_cache* host_copy, const kvq_cache* window,
                                    const int32_t* fetch_src, const int32_t* fetch_dst, int n_fetch,
                                    void* stream) {
  kvq_status st = check_cache(host_copy);
  if (st != KVQ_OK) return st;
  st = check_cache(window);
  if (st != KVQ_OK) return st;
  if (host_copy->fmt != window->fmt || host_copy->n_kv_heads != window->n_kv_heads ||
      host_copy->head_dim != window->head_dim || host_copy->block_size != window->block_size)
    return KVQ_ERR_ARG;
  if (n_fetch < 0) return KVQ_ERR_ARG;
  // Every run of the host copy must be memory the device can address at
  // the same address (pinned and mapped under unified addressing, or device
  // / managed memory).  Anything else is refused here rather than faulting
  // in a kernel.
  kvq_cache h = *host_copy;
  void** runs[4] = {&h.k_data, &h.v_data, &h.k_scales, &h.v_scales};
  const int n_runs = h.fmt == KVQ_F16 ? 2 : 4;
  for (int r = 0; r < n_runs; ++r) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, *runs[r]) != cudaSuccess) {
      (void)cudaGetLastError();
      return KVQ_ERR_ARG;
    }
    // the same address on both sides (unified addressing), so the appends
    // that write the host copy through this descriptor reach it too
    if (at.devicePointer == nullptr || at.devicePointer != *runs[r]) return KVQ_ERR_ARG;
  }
  if (n_fetch == 0) return KVQ_OK;
  if (fetch_src == nullptr || fetch_dst == nullptr || !aligned(fetch_src, 4) || !aligned(fetch_dst, 4))
    return KVQ_ERR_ARG;
  const cudaError_t e = launch_fetch(window->fmt, window->head_dim, &h, window, fetch_src,
                                     fetch_dst, n_fetch, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

KVQ_API const char* kvq_status_string(int status) {
  switch (status) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_ARG: return "KVQ_ERR_ARG: invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED: shape outside the implemented set";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE: workspace missing or too small";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA: CUDA launch error";
    default: return "unknown kvq_status";
  }
}

// ---------------------------------------------------------------------------
// kvq_decode_attn_static: decode attention for callers that cannot allocate.
//
// Some callers have no way to hand us a workspace: code that runs while a
// CUDA graph is being captured (cudaMalloc is not allowed there), plugins
// hosted by a framework whose allocator owns all device memory, and
// real-time loops whose memory is fixed once at start-up.  For them this
// entry point keeps its scratch in one file-scope device array of
// KVQ_STATIC_SCRATCH_BYTES, which exists on every device that loads the
// library for as long as the process lives.  The first call on a device
// (and the first after that device's context changes, e.g. after
// cudaDeviceReset) looks the array's device address up
// (cudaGetSymbolAddress) and caches it for that context; make that first
// call before any stream capture.  All calls share the array: two calls
// whose kernels overlap on the GPU (different streams, no ordering between
// them) race on it; the lock below covers only the address lookup.  Nothing
// in the array has to start at zero: the partial kernel writes every slot
// the combine kernel reads.
// ---------------------------------------------------------------------------
namespace kvq {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_STATIC_SCRATCH_BYTES];

ContextCache<void*> g_scratch_addr;

// Device address of g_decode_scratch in the current context.
kvq_status static_scratch_address(void** out) {
  const bool ok = per_context(g_scratch_addr, out, [](void** v) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return false;
    *v = p;
    return true;
  });
  return ok ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace
}  // namespace kvq

KVQ_API kvq_status kvq_decode_attn_static(const kvq_cache* cache, const float* q, int n_seq,
                                          int W, int n_q, const int32_t* ctx_lens, int max_ctx,
                                          const int32_t* block_table, int max_blocks_per_seq,
                                          float sm_scale, float* out, void* stream) {
  void* scratch = nullptr;
  const kvq_status st = kvq::static_scratch_address(&scratch);
  if (st != KVQ_OK) return st;
  // Same validation and kernels as kvq_decode_attn, with the split count
  // lowered until the plan fits the array; a request that does not fit even
  // with one split per (sequence, KV head) comes back as KVQ_ERR_WORKSPACE.
  return kvq::decode_impl(cache, q, n_seq, W, n_q, ctx_lens, max_ctx, block_table,
                          max_blocks_per_seq, sm_scale, out, scratch,
                          (size_t)KVQ_STATIC_SCRATCH_BYTES, stream, true);
}

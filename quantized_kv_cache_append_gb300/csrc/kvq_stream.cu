// kvq_stream.cu -- block streaming between a host copy of the pool and a
// resident window of device blocks.
//
// #711 kv: --kv k8v4 streams with --kv-resident, "What" and "How": the
// cache's authoritative copy lives in pinned host memory; a window of N
// cells' worth of device blocks holds the blocks a call reads; a block moves
// as its list of byte runs (K codes, K scales, V codes, V scales -- two runs
// for FP16), so every format streams through the same code; "Tests":
// attention over the streamed state equals attention over a fully resident
// pool, bit for bit (same bytes, same kernels, other block ids).
//
//   kvq_stream_plan   host only: which window slot serves each block a call
//                     reads, which blocks must be fetched, least recently
//                     used slots evicted first (state arrays owned by the
//                     caller).
//   kvq_stream_fetch  one kernel that reads the fetched blocks' runs
//                     straight from the host copy (mapped pinned memory,
//                     over the CPU-GPU link) and writes them into their
//                     slots: no copy engine, no per-run call.
#include <algorithm>
#include <vector>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

struct FetchArgs {
  const unsigned char* src[4];  // host copy runs (device-accessible)
  unsigned char* dst[4];        // window runs
  unsigned long long run_b[4];  // bytes of one block in each run (multiples of 16)
  int n_runs;
  const int32_t* fetch_src;     // [n_fetch] host block ids
  const int32_t* fetch_dst;     // [n_fetch] window slots
  int n_fetch;
  int n_src_blocks, n_dst_blocks;
  unsigned long long block_b;   // sum of run_b
};

// Thread i of the grid-stride walk copies 16-byte chunks i, i + stride, ...
// of the concatenation (fetch, run, byte); UNROLL chunks are loaded before
// any is stored, so each thread keeps several reads of host memory in
// flight.  Ids out of range skip the fetch.
template <int UNROLL>
__global__ void __launch_bounds__(256) fetch_kernel(FetchArgs a) {
  const unsigned long long chunks_per_block = a.block_b / 16;
  const unsigned long long total = chunks_per_block * (unsigned long long)a.n_fetch;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x * UNROLL;
  for (unsigned long long base = (unsigned long long)blockIdx.x * blockDim.x * UNROLL + threadIdx.x;
       base < total; base += stride) {
    uint4 v[UNROLL];
    unsigned char* to[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      to[u] = nullptr;
      const unsigned long long c = base + (unsigned long long)u * blockDim.x;
      if (c >= total) continue;
      const int f = (int)(c / chunks_per_block);
      unsigned long long off = (c - (unsigned long long)f * chunks_per_block) * 16;
      const int sb = a.fetch_src[f], db = a.fetch_dst[f];
      if (sb < 0 || sb >= a.n_src_blocks || db < 0 || db >= a.n_dst_blocks) continue;
      int r = 0;
      while (r + 1 < a.n_runs && off >= a.run_b[r]) {
        off -= a.run_b[r];
        ++r;
      }
      v[u] = *reinterpret_cast<const uint4*>(a.src[r] + (unsigned long long)sb * a.run_b[r] + off);
      to[u] = a.dst[r] + (unsigned long long)db * a.run_b[r] + off;
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u)
      if (to[u] != nullptr) *reinterpret_cast<uint4*>(to[u]) = v[u];
  }
}

}  // namespace

kvq_status stream_plan(int n_host_blocks, int n_slots, int32_t* slot_of_block, int32_t* block_of_slot,
                       int64_t* last_use, int64_t* clock, const int32_t* block_table, int n_seq,
                       int max_blocks, const int32_t* ctx_lens, int block_size, int32_t* slot_table,
                       int32_t* fetch_src, int32_t* fetch_dst, int* n_fetch, int* n_hits) {
  // the distinct host blocks this call reads, in first-use order (sorted
  // by id to drop repeats, then back into the order of first use: the cost
  // follows the blocks read, not the size of the host copy)
  std::vector<std::pair<int32_t, int32_t>> uses;  // (block, first use)
  for (int b = 0; b < n_seq; ++b) {
    const long long L = ctx_lens[b];
    if (L < 0 || L > (long long)max_blocks * block_size) return KVQ_ERR_ARG;
    const int nb = (int)((L + block_size - 1) / block_size);
    for (int j = 0; j < nb; ++j) {
      const int32_t blk = block_table[(size_t)b * max_blocks + j];
      if (blk >= 0 && blk < n_host_blocks) uses.emplace_back(blk, (int32_t)uses.size());
    }
  }
  std::sort(uses.begin(), uses.end());
  uses.erase(std::unique(uses.begin(), uses.end(),
                         [](const std::pair<int32_t, int32_t>& x, const std::pair<int32_t, int32_t>& y) {
                           return x.first == y.first;
                         }),
             uses.end());
  std::sort(uses.begin(), uses.end(),
            [](const std::pair<int32_t, int32_t>& x, const std::pair<int32_t, int32_t>& y) {
              return x.second < y.second;
            });
  std::vector<int32_t> need;
  need.reserve(uses.size());
  for (const auto& u : uses) need.push_back(u.first);
  if ((long long)need.size() > n_slots) return KVQ_ERR_UNSUPPORTED;  // nothing changed yet
  const int64_t now = ++*clock;
  int hits = 0;
  std::vector<int32_t> miss;
  for (int32_t blk : need) {
    const int32_t s = slot_of_block[blk];
    if (s >= 0 && s < n_slots && block_of_slot[s] == blk) {
      last_use[s] = now;
      ++hits;
    } else {
      slot_of_block[blk] = -1;
      miss.push_back(blk);
    }
  }
  // victims: free slots in index order, then the slots this call does not
  // read, least recently used first (ties: lower index)
  std::vector<int32_t> cand;
  for (int s = 0; s < n_slots; ++s)
    if (block_of_slot[s] < 0) cand.push_back(s);
  const size_t n_free = cand.size();
  for (int s = 0; s < n_slots; ++s)
    if (block_of_slot[s] >= 0 && last_use[s] != now) cand.push_back(s);
  std::stable_sort(cand.begin() + n_free, cand.end(),
                   [&](int32_t x, int32_t y) { return last_use[x] < last_use[y]; });
  for (size_t i = 0; i < miss.size(); ++i) {
    const int32_t s = cand[i];  // need.size() <= n_slots leaves enough candidates
    const int32_t old = block_of_slot[s];
    if (old >= 0 && old < n_host_blocks && slot_of_block[old] == s) slot_of_block[old] = -1;
    block_of_slot[s] = miss[i];
    slot_of_block[miss[i]] = s;
    last_use[s] = now;
    fetch_src[i] = miss[i];
    fetch_dst[i] = s;
  }
  *n_fetch = (int)miss.size();
  if (n_hits != nullptr) *n_hits = hits;
  // the window's block table: every entry of the rows, -1 where a block is
  // not resident (beyond a context, or an id out of range)
  for (int b = 0; b < n_seq; ++b)
    for (int j = 0; j < max_blocks; ++j) {
      const int32_t blk = block_table[(size_t)b * max_blocks + j];
      slot_table[(size_t)b * max_blocks + j] =
          (blk >= 0 && blk < n_host_blocks) ? slot_of_block[blk] : -1;
    }
  return KVQ_OK;
}

cudaError_t launch_fetch(int fmt, int hd, const kvq_cache* host, const kvq_cache* win,
                         const int32_t* fetch_src, const int32_t* fetch_dst, int n_fetch,
                         cudaStream_t s) {
  FetchArgs a = {};
  const unsigned long long rows = (unsigned long long)host->n_kv_heads * host->block_size;
  const int esz = fmt == KVQ_F16 ? 2 : 1;
  a.src[0] = static_cast<const unsigned char*>(host->k_data);
  a.dst[0] = static_cast<unsigned char*>(win->k_data);
  a.run_b[0] = rows * hd * esz;
  a.src[1] = static_cast<const unsigned char*>(host->v_data);
  a.dst[1] = static_cast<unsigned char*>(win->v_data);
  a.run_b[1] = rows * (fmt == KVQ_K8V4 ? hd / 2 : hd * esz);
  a.n_runs = 2;
  if (fmt != KVQ_F16) {
    a.src[2] = static_cast<const unsigned char*>(host->k_scales);
    a.dst[2] = static_cast<unsigned char*>(win->k_scales);
    a.run_b[2] = rows * (hd / kGroup) * 2;
    a.src[3] = static_cast<const unsigned char*>(host->v_scales);
    a.dst[3] = static_cast<unsigned char*>(win->v_scales);
    a.run_b[3] = rows * (fmt == KVQ_K8V4 ? hd / kQ4Block : hd / kGroup) * 2;
    a.n_runs = 4;
  }
  a.block_b = 0;
  for (int r = 0; r < a.n_runs; ++r) a.block_b += a.run_b[r];
  a.fetch_src = fetch_src;
  a.fetch_dst = fetch_dst;
  a.n_fetch = n_fetch;
  a.n_src_blocks = host->n_blocks;
  a.n_dst_blocks = win->n_blocks;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  constexpr int kUnroll = 4;
  const unsigned long long total = a.block_b / 16 * (unsigned long long)n_fetch;
  unsigned long long blocks = (total + 256 * kUnroll - 1) / (256 * kUnroll);
  const unsigned long long cap = (unsigned long long)(sms > 0 ? sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  fetch_kernel<kUnroll><<<(unsigned)blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq

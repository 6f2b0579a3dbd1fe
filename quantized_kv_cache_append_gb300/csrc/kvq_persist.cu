// kvq_persist.cu -- a sequence's cells gathered out of the paged pool into
// token-major runs, and scattered back.
//
// Path F format v3: persist per-head INT8 KV scales for INT8 + persistent
// KV interop, "Scope": what a saved turn keeps is its used cells' K/V bytes
// followed by their scales, token-major, and "Why": int8 bytes without the
// scales would hydrate to garbage, so int8 codes never move without them.
// #711 kv: --kv k8v4 streams with --kv-resident, "How": a block moves as its
// byte runs (codes, then scales).
//
// Runs: codes [n_cells][n_kv][hd] in the pool's element type, scales
// [n_cells][n_kv][hd/64] fp16 (int8 only); K8V4's V runs are its nibbles
// [n_cells][n_kv][hd/2] and scales [n_cells][n_kv][hd/32].  One thread
// moves 16 bytes of a row of K and the same 16 bytes of V (while the V row
// has them); the thread that takes a row's first chunk also moves its
// scales.  Loads and stores are coalesced along the
// row, then the KV heads, then the cells.  A block id out of range skips
// its cells (the gather leaves them unwritten, the scatter writes nothing).
#include "kvq_internal.cuh"

namespace kvq {
namespace {

// B bytes (2 .. 16, a power of two) from src to dst, both B-byte aligned
// (a row's scales: B = 2 per 64 or 32 dims, and rows start at multiples of
// B), as one access.
template <int B>
__device__ __forceinline__ void copy_run(void* dst, const void* src) {
  if constexpr (B == 16) *static_cast<uint4*>(dst) = __ldg(static_cast<const uint4*>(src));
  else if constexpr (B == 8) *static_cast<uint2*>(dst) = __ldg(static_cast<const uint2*>(src));
  else if constexpr (B == 4) *static_cast<uint32_t*>(dst) = __ldg(static_cast<const uint32_t*>(src));
  else *static_cast<unsigned short*>(dst) = __ldg(static_cast<const unsigned short*>(src));
}

template <int FMT, int HD, bool GATHER>
__global__ void __launch_bounds__(256) persist_kernel(PersistArgs a) {
  constexpr int ESZ = FMT == KVQ_F16 ? 2 : 1;
  constexpr int KROWB = HD * ESZ;                             // K row bytes
  constexpr int VROWB = FMT == KVQ_K8V4 ? HD / 2 : KROWB;     // V row bytes
  constexpr int CPR = KROWB / 16;  // 16-byte chunks per row (K, the longer one)
  constexpr int NG = HD / kGroup;
  constexpr int NVS = FMT == KVQ_K8V4 ? HD / kQ4Block : NG;  // V scales per row
  const long long rows = (long long)a.n_cells * a.pool.n_kv;
  const long long total = rows * CPR;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int bs = 1 << a.pool.bs_log2;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int chunk = (int)(i % CPR);
    const long long r = i / CPR;  // p * n_kv + kvh (token-major)
    const int p = (int)(r / a.pool.n_kv);
    const int kvh = (int)(r - (long long)p * a.pool.n_kv);
    const int blk = __ldg(a.block_row + (p >> a.pool.bs_log2));
    if (blk < 0 || blk >= a.pool.n_blocks) continue;
    const size_t row = ((size_t)blk * a.pool.n_kv + kvh) * bs + (p & (bs - 1));
    const size_t pool_off = row * KROWB + (size_t)chunk * 16;
    const size_t run_off = (size_t)r * KROWB + (size_t)chunk * 16;
    const size_t vpool_off = row * VROWB + (size_t)chunk * 16;
    const size_t vrun_off = (size_t)r * VROWB + (size_t)chunk * 16;
    const bool v_here = chunk * 16 < VROWB;
    if constexpr (GATHER) {
      *reinterpret_cast<uint4*>(static_cast<char*>(a.codes_k) + run_off) =
          __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.pool.k) + pool_off));
      if (v_here)
        *reinterpret_cast<uint4*>(static_cast<char*>(a.codes_v) + vrun_off) =
            __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.pool.v) + vpool_off));
    } else {
      *reinterpret_cast<uint4*>(static_cast<char*>(a.pool_k) + pool_off) =
          __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.codes_k) + run_off));
      if (v_here)
        *reinterpret_cast<uint4*>(static_cast<char*>(a.pool_v) + vpool_off) =
            __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.codes_v) + vrun_off));
    }
    if constexpr (FMT != KVQ_F16) {
      if (chunk == 0) {  // a row's scales, each run as one aligned vector
        if constexpr (GATHER) {
          copy_run<NG * 2>(a.scales_k + (size_t)r * NG, a.pool.ks + row * NG);
          copy_run<NVS * 2>(a.scales_v + (size_t)r * NVS, a.pool.vs + row * NVS);
        } else {
          copy_run<NG * 2>(a.pool_ks + row * NG, a.scales_k + (size_t)r * NG);
          copy_run<NVS * 2>(a.pool_vs + row * NVS, a.scales_v + (size_t)r * NVS);
        }
      }
    }
  }
}

template <int FMT, bool GATHER>
cudaError_t launch_fmt(int hd, const PersistArgs& a, cudaStream_t s, int blocks) {
  switch (hd) {
    case 64: persist_kernel<FMT, 64, GATHER><<<blocks, 256, 0, s>>>(a); break;
    case 128: persist_kernel<FMT, 128, GATHER><<<blocks, 256, 0, s>>>(a); break;
    case 256: persist_kernel<FMT, 256, GATHER><<<blocks, 256, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_persist(int fmt, int hd, bool gather, const PersistArgs& a, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int esz = fmt == KVQ_F16 ? 2 : 1;
  const long long total = (long long)a.n_cells * a.pool.n_kv * (hd * esz / 16);
  long long blocks = (total + 255) / 256;
  // FP16 rows: one 16-byte chunk a thread over a grid that holds them all
  // (measured 8 % faster); int8 and K8V4 rows, whose first chunk also moves
  // the scales: grid-stride beyond 8 CTAs an SM (measured 5-12 % faster)
  const long long cap = fmt == KVQ_F16 ? 0x7fffffffLL : (long long)(sms > 0 ? sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (fmt == KVQ_F16)
    return gather ? launch_fmt<KVQ_F16, true>(hd, a, s, (int)blocks)
                  : launch_fmt<KVQ_F16, false>(hd, a, s, (int)blocks);
  if (fmt == KVQ_Q8)
    return gather ? launch_fmt<KVQ_Q8, true>(hd, a, s, (int)blocks)
                  : launch_fmt<KVQ_Q8, false>(hd, a, s, (int)blocks);
  if (fmt == KVQ_K8V4)
    return gather ? launch_fmt<KVQ_K8V4, true>(hd, a, s, (int)blocks)
                  : launch_fmt<KVQ_K8V4, false>(hd, a, s, (int)blocks);
  return cudaErrorInvalidValue;
}

}  // namespace kvq

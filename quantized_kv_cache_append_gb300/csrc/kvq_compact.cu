// kvq_compact.cu -- copy one sequence's cells out to contiguous FP16 staging.
//
// #3084 qwen35: FP16 K/V cache by default, int8 with --kv-q8, "Extra Notes":
// k_kv_f16 compacts [kvh][ctx][HD] into the [kvh][P][HD] halves that the
// prompt chunk's QK^T and PV products read; with an FP16 cache it becomes a
// pure copy ("What changed").  With the int8 cache each value is written as
// fp16(code * scale); the product of an 8-bit code and an fp16 scale is
// exact in fp32, so the only rounding is __float2half_rn (nearest even).
//
// One thread moves 8 consecutive dims of one row: 8 int8 codes (8 bytes) or
// 8 fp16 values (16 bytes) in, 16 bytes out.  Consecutive threads walk the
// dims of a row, then the cells, so loads and stores are both coalesced.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

template <int FMT, int HD>
__global__ void __launch_bounds__(256) compact_kernel(CompactArgs a) {
  constexpr int CPR = HD / 8;  // 8-dim chunks per row
  constexpr int NG = HD / kGroup;
  const long long total = 2LL * a.pool.n_kv * a.n_cells * CPR;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int bs = 1 << a.pool.bs_log2;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int chunk = (int)(i % CPR);
    const long long r = i / CPR;                 // (which, kvh, p)
    const int p = (int)(r % a.n_cells);
    const long long wk = r / a.n_cells;          // which * n_kv + kvh
    const int kvh = (int)(wk % a.pool.n_kv);
    const int which = (int)(wk / a.pool.n_kv);   // 0 = K, 1 = V

    const int blk = __ldg(a.block_row + (p >> a.pool.bs_log2));
    if (blk < 0 || blk >= a.pool.n_blocks) continue;  // precondition broken: skip
    const size_t row = ((size_t)blk * a.pool.n_kv + kvh) * bs + (p & (bs - 1));
    __half* dst = (which ? a.out_v : a.out_k) + ((size_t)kvh * a.n_cells + p) * HD + chunk * 8;

    if constexpr (FMT == KVQ_F16) {
      const __half* src = static_cast<const __half*>(which ? a.pool.v : a.pool.k) + row * HD;
      *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src + chunk * 8));
    } else {
      const int8_t* src = static_cast<const int8_t*>(which ? a.pool.v : a.pool.k) + row * HD;
      const __half* sc = (which ? a.pool.vs : a.pool.ks) + row * NG;
      const uint2 codes = __ldg(reinterpret_cast<const uint2*>(src + chunk * 8));
      const float sf = __half2float(sc[(chunk * 8) / kGroup]);
      uint32_t outw[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const uint32_t w = e < 4 ? codes.x : codes.y;
        const int sh = (e & 3) * 8;
        const float lo = (float)(int8_t)(w >> sh) * sf;
        const float hi = (float)(int8_t)(w >> (sh + 8)) * sf;
        outw[e / 2] = (uint32_t)__half_as_ushort(__float2half_rn(lo)) |
                      ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
      }
      *reinterpret_cast<uint4*>(dst) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
    }
  }
}

template <int FMT>
cudaError_t launch_fmt(int hd, const CompactArgs& a, cudaStream_t s, int blocks) {
  switch (hd) {
    case 64: compact_kernel<FMT, 64><<<blocks, 256, 0, s>>>(a); break;
    case 128: compact_kernel<FMT, 128><<<blocks, 256, 0, s>>>(a); break;
    case 256: compact_kernel<FMT, 256><<<blocks, 256, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compact(int fmt, int hd, const CompactArgs& a, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long total = 2LL * a.pool.n_kv * a.n_cells * (hd / 8);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)(sms > 0 ? sms : 1) * 8;  // grid-stride beyond 8 CTAs/SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return fmt == KVQ_F16 ? launch_fmt<KVQ_F16>(hd, a, s, (int)blocks)
                        : launch_fmt<KVQ_Q8>(hd, a, s, (int)blocks);
}

}  // namespace kvq

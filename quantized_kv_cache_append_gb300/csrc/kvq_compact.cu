// kvq_compact.cu -- copy one sequence's cells out to contiguous FP16 staging.
//
// #3084 qwen35: FP16 K/V cache by default, int8 with --kv-q8, "Extra Notes":
// k_kv_f16 compacts [kvh][ctx][HD] into the [kvh][P][HD] halves that the
// prompt chunk's QK^T and PV products read; with an FP16 cache it becomes a
// pure copy ("What changed").  With the int8 cache each value is written as
// fp16(code * scale); the product of an 8-bit code and an fp16 scale is
// exact in fp32, so the only rounding is __float2half_rn (nearest even).
//
// FP16: grid y = (K or V, KV head), grid-stride, one thread copies 8 dims
// (16 bytes).  int8: CTA x of KV head y takes the cells [x C, x C + C),
// C = 256 / (HD / 16), one thread one 16-code chunk of K and the same chunk
// of V (both loads issued first); it widens each code exactly to fp16 (XOR
// 0x80, PRMT with the 0x64 exponent byte, minus 1152) and multiplies pairs
// by the group's fp16 scale with mul.rn.f16x2: the product of a code and an
// fp16 scale is exact, and the fp16 multiply rounds it once to nearest
// even, with subnormals, which is fp16(code * scale).  Loads and stores are
// coalesced along the dims of a row, then the cells.
//
// K8V4 (#711 kv: --kv k8v4 streams with --kv-resident, "What": INT8 K +
// rotated Q4_0 V): the same CTAs take K as the int8 format, then V rows:
// decoded in the rotated basis, (code - 8) * d (exact in fp32), rotated
// back by the same fp32 butterflies as the append's rotation (wht_group),
// divided by head_dim (a power of two, exact; applied to d first, which
// gives the same bits since scaling by a power of two commutes with every
// rounded sum) and rounded to fp16.  A V row is held by a group of lanes;
// the K chunks (memory-bound) and the V rows (ALU-bound) of different CTAs
// overlap on an SM.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// (fp16_rne(lo), fp16_rne(hi)) packed, one conversion
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Codes in bytes 0, 1 (sel 0x4140) or 2, 3 (sel 0x4342) of w, times scale s2.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t w, uint32_t sel, uint32_t s2) {
  const uint32_t biased = w ^ 0x80808080u;  // c + 128 as unsigned bytes
  const uint32_t h = hsub2(prmt(biased, 0x64646464u, sel), 0x64806480u);  // (1024 + u) - 1152 = c
  return hmul2(h, s2);
}

// int8 codes of chunk `chunk` (16 dims) of cell p of KV head kvh, K (which
// 0) or V (1), widened and scaled to fp16 into the staging; a block id out
// of range skips the cell.
template <int HD>
__device__ __forceinline__ void q8_chunk(const CompactArgs& a, int kvh, int which, int p, int chunk) {
  constexpr int DPT = 16, NG = HD / kGroup;
  const int blk = __ldg(a.block_row + (p >> a.pool.bs_log2));
  if (blk < 0 || blk >= a.pool.n_blocks) return;  // precondition broken: skip
  const int bs = 1 << a.pool.bs_log2;
  const size_t row = ((size_t)blk * a.pool.n_kv + kvh) * bs + (p & (bs - 1));
  __half* dst = (which ? a.out_v : a.out_k) + ((size_t)kvh * a.n_cells + p) * HD + chunk * DPT;
  const int8_t* src = static_cast<const int8_t*>(which ? a.pool.v : a.pool.k) + row * HD;
  const uint4 c = __ldg(reinterpret_cast<const uint4*>(src + chunk * DPT));
  const unsigned short sbits =
      __half_as_ushort(((which ? a.pool.vs : a.pool.ks) + row * NG)[(chunk * DPT) / kGroup]);
  const uint32_t s2 = (uint32_t)sbits * 0x10001u;
  uint4 o0, o1;
  o0.x = dequant_pair(c.x, 0x4140u, s2);
  o0.y = dequant_pair(c.x, 0x4342u, s2);
  o0.z = dequant_pair(c.y, 0x4140u, s2);
  o0.w = dequant_pair(c.y, 0x4342u, s2);
  o1.x = dequant_pair(c.z, 0x4140u, s2);
  o1.y = dequant_pair(c.z, 0x4342u, s2);
  o1.z = dequant_pair(c.w, 0x4140u, s2);
  o1.w = dequant_pair(c.w, 0x4342u, s2);
  reinterpret_cast<uint4*>(dst)[0] = o0;
  reinterpret_cast<uint4*>(dst)[1] = o1;
}

// int8 compaction: CTA x of KV head y takes cells [x C, x C + C) with
// C = 256 / (HD / 16); each thread widens one 16-code chunk of K and the
// same chunk of V, both loads issued before either conversion.
template <int HD>
__global__ void __launch_bounds__(256) compact_q8_kernel(CompactArgs a) {
  constexpr int CPR = HD / 16, C = 256 / CPR, NG = HD / kGroup;
  const int kvh = blockIdx.y;
  const int p = blockIdx.x * C + threadIdx.x / CPR, chunk = threadIdx.x % CPR;
  if (p >= a.n_cells) return;  // no barrier in this kernel
  const int blk = __ldg(a.block_row + (p >> a.pool.bs_log2));
  if (blk < 0 || blk >= a.pool.n_blocks) return;  // precondition broken: skip
  const int bs = 1 << a.pool.bs_log2;
  const size_t row = ((size_t)blk * a.pool.n_kv + kvh) * bs + (p & (bs - 1));
  const size_t co = row * HD + chunk * 16, so = row * NG + (chunk * 16) / kGroup;
  const uint4 ck = __ldg(reinterpret_cast<const uint4*>(static_cast<const int8_t*>(a.pool.k) + co));
  const uint4 cv = __ldg(reinterpret_cast<const uint4*>(static_cast<const int8_t*>(a.pool.v) + co));
  const uint32_t sk = (uint32_t)__half_as_ushort(a.pool.ks[so]) * 0x10001u;
  const uint32_t sv = (uint32_t)__half_as_ushort(a.pool.vs[so]) * 0x10001u;
  const size_t out = ((size_t)kvh * a.n_cells + p) * HD + chunk * 16;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint4 c = which ? cv : ck;
    const uint32_t s2 = which ? sv : sk;
    uint4 o0, o1;
    o0.x = dequant_pair(c.x, 0x4140u, s2);
    o0.y = dequant_pair(c.x, 0x4342u, s2);
    o0.z = dequant_pair(c.y, 0x4140u, s2);
    o0.w = dequant_pair(c.y, 0x4342u, s2);
    o1.x = dequant_pair(c.z, 0x4140u, s2);
    o1.y = dequant_pair(c.z, 0x4342u, s2);
    o1.z = dequant_pair(c.w, 0x4140u, s2);
    o1.w = dequant_pair(c.w, 0x4342u, s2);
    uint4* dst = reinterpret_cast<uint4*>((which ? a.out_v : a.out_k) + out);
    dst[0] = o0;
    dst[1] = o1;
  }
}

// K8V4 V rows: a cell's row is held by a group of LPR = HD / VPL lanes
// (VPL consecutive dims each, within one 32-dim block), so a warp
// de-rotates RPW = 32 / LPR cells at once.
template <int HD>
struct V4Rows {
  static constexpr int VPL = HD >= 128 ? 16 : 8;
  static constexpr int LPR = HD / VPL;
  static constexpr int RPW = 32 / LPR;
};

// The warp's RPW cells from p_base (lane group g takes cell p_base + g);
// cells past the end or in an out-of-range block are skipped, every lane
// still taking part in the shuffles.
template <int HD>
__device__ __forceinline__ void v4_rows(const CompactArgs& a, int kvh, int p_base, int lane) {
  constexpr int VPL = V4Rows<HD>::VPL, LPR = V4Rows<HD>::LPR;
  constexpr int NB = HD / kQ4Block;
  const int j = lane & (LPR - 1);
  const int bs = 1 << a.pool.bs_log2;
  const int p = p_base + lane / LPR;
  const int blk = p < a.n_cells ? __ldg(a.block_row + (p >> a.pool.bs_log2)) : -1;
  const bool ok = blk >= 0 && blk < a.pool.n_blocks;
  float x[VPL];
  if (ok) {
    const size_t row = ((size_t)blk * a.pool.n_kv + kvh) * bs + (p & (bs - 1));
    const unsigned char* src = static_cast<const unsigned char*>(a.pool.v) + row * (HD / 2) + j * (VPL / 2);
    // d / HD: the power-of-two factor of the inverse rotation, taken
    // before the butterflies (exact, and it commutes with every sum)
    const float d = __half2float(__ldg(a.pool.vs + row * NB + (j * VPL) / kQ4Block)) * (1.0f / HD);
    uint32_t w[VPL / 8];
    if constexpr (VPL == 16) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
      w[0] = u.x;
      w[VPL / 8 > 1 ? 1 : 0] = u.y;
    } else {
      w[0] = __ldg(reinterpret_cast<const uint32_t*>(src));
    }
#pragma unroll
    for (int e = 0; e < VPL; ++e) {
      // 2^23 + code as float bits, minus 2^23 + 8: code - 8, exactly
      const float c = __uint_as_float(0x4b000000u | ((w[e / 8] >> (4 * (e % 8))) & 15u)) - 8388616.0f;
      x[e] = __fmul_rn(c, d);
    }
  } else {
#pragma unroll
    for (int e = 0; e < VPL; ++e) x[e] = 0.f;
  }
  wht_group<VPL, LPR>(x, lane);
  if (ok) {
    __half* dst = a.out_v + ((size_t)kvh * a.n_cells + p) * HD + j * VPL;
#pragma unroll
    for (int q = 0; q < VPL / 8; ++q)
      reinterpret_cast<uint4*>(dst)[q] =
          make_uint4(f16x2_rn(x[8 * q], x[8 * q + 1]), f16x2_rn(x[8 * q + 2], x[8 * q + 3]),
                     f16x2_rn(x[8 * q + 4], x[8 * q + 5]), f16x2_rn(x[8 * q + 6], x[8 * q + 7]));
  }
}

// K8V4 compaction in one launch: CTA x of KV head y takes cells
// [x C, x C + C) with C = 256 / (HD / 16): first every thread one 16-code
// chunk of K (memory-bound), then the warps the V rows in lane groups
// (ALU-bound), so the two kinds of work of different CTAs overlap on an SM.
template <int HD>
__global__ void __launch_bounds__(256) compact_k8v4_kernel(CompactArgs a) {
  constexpr int CPR = HD / 16;              // K chunks per cell
  constexpr int C = 256 / CPR;              // cells per CTA
  constexpr int RPW = V4Rows<HD>::RPW;
  const int kvh = blockIdx.y;
  const int c0 = blockIdx.x * C;
  const int pk = c0 + threadIdx.x / CPR;
  if (pk < a.n_cells) q8_chunk<HD>(a, kvh, 0, pk, threadIdx.x % CPR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int it = 0; it < C / (8 * RPW); ++it) {
    const int p_base = c0 + (it * 8 + warp) * RPW;
    if (p_base < a.n_cells) v4_rows<HD>(a, kvh, p_base, lane);  // warp-uniform
  }
}

// FP16 compaction: a pure copy, grid-stride over (cell, 16-byte chunk),
// grid y = (K or V, KV head).
template <int HD>
__global__ void __launch_bounds__(256) compact_f16_kernel(CompactArgs a) {
  constexpr int DPT = 8;          // dims per thread (16 bytes)
  constexpr int CPR = HD / DPT;   // threads per row
  const int kvh = blockIdx.y % a.pool.n_kv;
  const int which = blockIdx.y / a.pool.n_kv;    // 0 = K, 1 = V
  const long long total = (long long)a.n_cells * CPR;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int bs = 1 << a.pool.bs_log2;
  __half* out = which ? a.out_v : a.out_k;
  const __half* pool = static_cast<const __half*>(which ? a.pool.v : a.pool.k);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int p = (int)(i / CPR);
    const int chunk = (int)(i % CPR);
    const int blk = __ldg(a.block_row + (p >> a.pool.bs_log2));
    if (blk < 0 || blk >= a.pool.n_blocks) continue;  // precondition broken: skip
    const size_t row = ((size_t)blk * a.pool.n_kv + kvh) * bs + (p & (bs - 1));
    __half* dst = out + ((size_t)kvh * a.n_cells + p) * HD + chunk * DPT;
    *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(pool + row * HD + chunk * DPT));
  }
}

}  // namespace

cudaError_t launch_compact(int fmt, int hd, const CompactArgs& a, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  if (fmt != KVQ_F16) {  // one thread a 16-code chunk: CTAs of 256 / (HD / 16) cells per KV head
    const int cells = 256 / (hd / 16);
    long long xs = (a.n_cells + cells - 1) / cells;
    if (xs > 0x7fffffffLL || a.pool.n_kv > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)xs, (unsigned)a.pool.n_kv);
    const bool q8 = fmt == KVQ_Q8;
    switch (hd) {
      case 64: q8 ? compact_q8_kernel<64><<<grid, 256, 0, s>>>(a) : compact_k8v4_kernel<64><<<grid, 256, 0, s>>>(a); break;
      case 128: q8 ? compact_q8_kernel<128><<<grid, 256, 0, s>>>(a) : compact_k8v4_kernel<128><<<grid, 256, 0, s>>>(a); break;
      case 256: q8 ? compact_q8_kernel<256><<<grid, 256, 0, s>>>(a) : compact_k8v4_kernel<256><<<grid, 256, 0, s>>>(a); break;
      default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  const long long per_row = (long long)a.n_cells * (hd / 8);  // threads per (K or V, KV head)
  const int ys = 2 * a.pool.n_kv;
  long long xs = (per_row + 255) / 256;
  const long long cap = ((long long)sms * 8 + ys - 1) / ys;  // about 8 CTAs per SM in total
  if (xs > cap) xs = cap;
  if (xs < 1) xs = 1;
  if (ys > 65535) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)xs, (unsigned)ys);
  switch (hd) {
    case 64: compact_f16_kernel<64><<<grid, 256, 0, s>>>(a); break;
    case 128: compact_f16_kernel<128><<<grid, 256, 0, s>>>(a); break;
    case 256: compact_f16_kernel<256><<<grid, 256, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace kvq

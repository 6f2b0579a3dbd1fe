// kvq_append.cu -- quantize-on-write of new K/V rows into the paged pool.
//
// #3084 qwen35: FP16 K/V cache by default, int8 with --kv-q8, "What changed":
// under --kv-q8 a row is written as scale = fp16(max|x| / 127) per 64 dims and
// code = clamp(rint(x / scale), -127, 127); the FP16 cache stores fp16(x).
// The same section notes that the group maximum needs every thread to reach
// a barrier before the stores.  Here the lanes of a 64-dim group (a quad
// for a few tokens; 4 lanes of 16 dims each for bulk appends) take the
// group maximum by a warp-shuffle butterfly that every lane executes: no
// __syncthreads exists in these kernels and no early return can skip one.
//
// Bit-exactness: max|x| is exact; a / 127 and x / s are the IEEE fp32
// quotients the pages define (the library is built without fast-math, so
// '/' is div.rn.f32), replaced by multiplies only where those provably give
// the same fp16 scale (group_scale) or the same integer code (codes4);
// __float2half_rn rounds to nearest even with subnormals; rounding is to
// nearest even, and clamping before rounding equals clamping after it for
// the bound 127.
//
// #711 kv: --kv k8v4 streams with --kv-resident, "What": K8V4 keeps K as the
// int8 format does and V rotated, as Q4_0 (one fp16 scale per 32 dims,
// 4-bit codes with an offset of 8).  The rotation is the Walsh-Hadamard
// transform in fp32 butterflies, stage by stage, and the codes follow the
// same bit-exact discipline as the int8 ones.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

// The group scale fp16_rne(fl32(a / 127)) from a multiply: y = a * fl(1/127)
// is within 2 fp32 ulps of fl32(a / 127), so the two round to the same fp16
// value unless an fp16 rounding midpoint (13 discarded bits equal to 0x1000)
// lies within that distance, or the result leaves the fp16 normal range;
// only then is the quotient itself computed.
__device__ __forceinline__ __half group_scale(float a) {
  const float y = a * (1.0f / 127.0f);
  const uint32_t low = __float_as_uint(y) & 0x1fffu;
  const bool exact_needed = (low > 0x1000u - 4u && low < 0x1000u + 4u) || !(y >= 6.103515625e-05f) ||
                            !(y < 65504.0f);
  return __float2half_rn(exact_needed ? a / 127.0f : y);
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Packed fp32 pairs (two lanes of work per instruction).
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  return ((unsigned long long)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo2(unsigned long long v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(unsigned long long v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// The int8 code clamp(rint(x / sf), -127, 127) from the IEEE fp32 quotient
// itself, as a byte (0 for a zero scale or a NaN quotient).
__device__ __forceinline__ uint32_t exact_code(float x, float sf) {
  if (sf == 0.0f) return 0u;
  const float qv = x / sf;
  if (!(qv == qv)) return 0u;
  return (uint32_t)(int)fminf(fmaxf(rintf(qv), -127.0f), 127.0f) & 0xffu;
}

// Codes of 4 values of one group (finite group maximum, so x is finite), as
// 4 bytes.  y = x * rs (rs = 1 / sf within one ulp) is within 2^-21 |x / sf|
// of the real quotient, and |x / sf| < 256, so wherever y lies more than
// 2.5e-4 from a half-integer the real quotient, its fp32 rounding and y
// round to the same integer; only inside that band are the quotients
// themselves used.  After clamping y to [-127, 127], y + 1.5 * 2^23 rounds y
// to an integer (to nearest, ties to even) in the low mantissa bits, whose
// low byte is the two's-complement code.
__device__ __forceinline__ uint32_t codes4(const float4& x, float sf, float rs) {
  if (sf == 0.0f) return 0u;
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  const unsigned long long r2 = pack2(rs, rs), m2 = pack2(kMagic, kMagic);
  const unsigned long long p01 = mul2(pack2(x.x, x.y), r2), p23 = mul2(pack2(x.z, x.w), r2);
  const unsigned long long y01 = pack2(fminf(fmaxf(lo2(p01), -127.0f), 127.0f),
                                       fminf(fmaxf(hi2(p01), -127.0f), 127.0f));
  const unsigned long long y23 = pack2(fminf(fmaxf(lo2(p23), -127.0f), 127.0f),
                                       fminf(fmaxf(hi2(p23), -127.0f), 127.0f));
  const unsigned long long t01 = add2(y01, m2), t23 = add2(y23, m2);
  const unsigned long long d01 = sub2(y01, sub2(t01, m2)), d23 = sub2(y23, sub2(t23, m2));
  constexpr float kBand = 0.5f - 2.5e-4f;
  const bool tie = fabsf(lo2(d01)) > kBand || fabsf(hi2(d01)) > kBand || fabsf(lo2(d23)) > kBand ||
                   fabsf(hi2(d23)) > kBand;
  if (tie)  // near a tie: the quotients decide (a few groups in a thousand)
    return exact_code(x.x, sf) | (exact_code(x.y, sf) << 8) | (exact_code(x.z, sf) << 16) |
           (exact_code(x.w, sf) << 24);
  return prmt(prmt((uint32_t)t01, (uint32_t)(t01 >> 32), 0x0040u),
              prmt((uint32_t)t23, (uint32_t)(t23 >> 32), 0x0040u), 0x5410u);
}

// Destination row of row index `row` (= token * n_kv + kvh): the token's
// sequence, position and block-table entry; -1 when a precondition is
// broken (then nothing is written).
__device__ __forceinline__ long long dest_row(const AppendArgs& a, long long row, bool rows32) {
  int tok, kvh;
  if (rows32) {  // 32-bit division where the row count fits
    tok = (int)((unsigned)row / (unsigned)a.n_kv);
    kvh = (int)row - tok * a.n_kv;
  } else {
    tok = (int)(row / a.n_kv);
    kvh = (int)(row - (long long)tok * a.n_kv);
  }
  const int seq = __ldg(a.tok_seq + tok);
  const int pos = __ldg(a.tok_pos + tok);
  if (seq < 0 || seq >= a.n_seq || pos < 0 || (pos >> a.bs_log2) >= a.max_blocks) return -1;
  const int blk = __ldg(a.block_table + (size_t)seq * a.max_blocks + (pos >> a.bs_log2));
  if (blk < 0 || blk >= a.n_blocks) return -1;
  return ((long long)blk * a.n_kv + kvh) * (1LL << a.bs_log2) + (pos & ((1 << a.bs_log2) - 1));
}

// FP16 append.  The K and V inputs are flat arrays of n_tok * n_kv * HD
// floats, read as 16-byte chunks; each thread handles U chunk positions of
// K and the same positions of V (2U loads in flight before the first use),
// warp j of the grid covering chunks [32 U j, 32 U (j + 1)); W warps a CTA.
template <int HD, int U, int W>
__global__ void __launch_bounds__(W * 32) append_f16_kernel(AppendArgs a) {
  constexpr int CPR = HD / 4;  // 16-byte chunks per row
  // Launched as a programmatic dependent: wait for the previous kernel's
  // writes (k, v, positions may come from it), then let the next kernel's
  // launch begin.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long n_chunks = (long long)a.n_tok * a.n_kv * CPR;
  const bool rows32 = n_chunks / CPR <= 0x7fffffffLL;
  const long long base = ((long long)blockIdx.x * W + (threadIdx.x >> 5)) * 32LL * U;
  const float4* k4 = reinterpret_cast<const float4*>(a.k);
  const float4* v4 = reinterpret_cast<const float4*>(a.v);

  float4 xk[U], xv[U];
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const long long f = base + 32LL * j + lane;
    xk[j] = xv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (f < n_chunks) {
      xk[j] = __ldcs(k4 + f);
      xv[j] = __ldcs(v4 + f);
    }
  }
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const long long f = base + 32LL * j + lane;
    if (f >= n_chunks) continue;
    const long long dr = dest_row(a, f / CPR, rows32);
    if (dr < 0) continue;
    const int d = (int)(f % CPR) * 4;  // first dim of this chunk
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const float4 x = which ? xv[j] : xk[j];
      __half* dst = static_cast<__half*>(which ? a.v_dst : a.k_dst) + dr * HD + d;
      uint2 u;
      u.x = (uint32_t)__half_as_ushort(__float2half_rn(x.x)) |
            ((uint32_t)__half_as_ushort(__float2half_rn(x.y)) << 16);
      u.y = (uint32_t)__half_as_ushort(__float2half_rn(x.z)) |
            ((uint32_t)__half_as_ushort(__float2half_rn(x.w)) << 16);
      *reinterpret_cast<uint2*>(dst) = u;
    }
  }
}

// int8 append for a few tokens (decode steps; bulk appends use
// append_q8_rows_kernel).  A quad of 4 lanes owns one 64-dim group of one row: lane q
// holds the 16-byte chunks q, q + 4, q + 8, q + 12 of the group (dims
// 16 i + 4 q .. + 3), so every load instruction reads 64 contiguous bytes
// per quad.  The group maximum is a 2-step butterfly inside the quad (on
// the bit patterns of |x|, whose integer order is the numeric order with
// inf and NaN on top); scale, reciprocal and 16 codes follow per lane.
// Each thread handles U groups of K and the same groups of V; a warp covers
// 8 U groups, W warps a CTA.  With KV_SPLIT (few tokens) even warps take K
// and odd warps V, halving each thread's chain.
template <int HD, int U, int W, bool KV_SPLIT>
__global__ void __launch_bounds__(W * 32) append_q8_kernel(AppendArgs a) {
  constexpr int NG = HD / kGroup;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31, q = lane & 3, quad = lane >> 2;
  const long long n_groups = (long long)a.n_tok * a.n_kv * NG;
  const bool rows32 = n_groups / NG <= 0x7fffffffLL;
  const long long wid = (long long)blockIdx.x * W + (threadIdx.x >> 5);
  const int only = KV_SPLIT ? (int)(wid & 1) : -1;  // K (0) or V (1) only, or both (-1)
  const long long gbase = (KV_SPLIT ? wid >> 1 : wid) * 8LL * U + quad;
  const float4* k4 = reinterpret_cast<const float4*>(a.k);
  const float4* v4 = reinterpret_cast<const float4*>(a.v);

  float4 x[2][U][4];  // [K, V][group][chunk]
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const long long g = gbase + 8LL * u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[0][u][i] = x[1][u][i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g < n_groups) {
        if (only != 1) x[0][u][i] = __ldcs(k4 + g * 16 + 4 * i + q);
        if (only != 0) x[1][u][i] = __ldcs(v4 + g * 16 + 4 * i + q);
      }
    }
  }
  long long dr[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const long long g = gbase + 8LL * u;
    dr[u] = g < n_groups ? dest_row(a, g / NG, rows32) : -1;
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const long long g = gbase + 8LL * u;
    const int gi = (int)(g % NG);
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      if (KV_SPLIT && which != only) continue;  // warp-uniform
      uint32_t mb = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4& v = x[which][u][i];
        mb = max(mb, max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                         max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu)));
      }
      // every lane takes part (quads past the end carry zeros, store nothing)
      mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      const float amax = __uint_as_float(mb);
      const __half sh = group_scale(amax);
      const float sf = __half2float(sh);
      if (dr[u] < 0) continue;
      int8_t* dst = static_cast<int8_t*>(which ? a.v_dst : a.k_dst) + dr[u] * HD + gi * kGroup + 4 * q;
      if (amax <= 3.4028234663852886e38f) {  // finite group: packed fast path
        const float rs = rcp_approx(sf);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint32_t*>(dst + 16 * i) = codes4(x[which][u][i], sf, rs);
      } else {  // inf or NaN in the group: element by element from the quotients
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4& v = x[which][u][i];
          *reinterpret_cast<uint32_t*>(dst + 16 * i) = exact_code(v.x, sf) | (exact_code(v.y, sf) << 8) |
                                                        (exact_code(v.z, sf) << 16) |
                                                        (exact_code(v.w, sf) << 24);
        }
      }
      if (q == 0) (which ? a.vs_dst : a.ks_dst)[dr[u] * NG + gi] = sh;
    }
  }
}

// K8V4 V codes of U values y of one block of scale d: the 4-bit offset
// codes clamp(rint(y / d), -8, 7) + 8, packed 4 bits each (value e in bits
// 4e..4e+3).  |y / d| <= 8 (up to d's fp16 rounding), so y * rs (rs ~ 1/d)
// is within 2e-6 of the quotient and decides the integer wherever it lies
// more than 2.5e-4 from a half-integer; adding and taking off 1.5 * 2^23
// rounds it (to nearest even) in packed pairs.  If any of the U values
// lies inside that band, or is not finite, the IEEE quotients decide all
// U (a NaN quotient gives 0).  Clamping to integer bounds commutes with
// rounding; the clamped integer k plus 1.5 * 2^23 + 8 has k + 8 in its
// low mantissa bits.  d == 0 gives code 8 throughout.
template <int U>
__device__ __forceinline__ uint32_t q4_codes(const float (&y)[U], float d) {
  if (d == 0.0f) return U == 4 ? 0x8888u : 0x88u;
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  constexpr float kBand = 0.5f - 2.5e-4f;
  const float rs = rcp_approx(d);
  const unsigned long long r2 = pack2(rs, rs), m2 = pack2(kMagic, kMagic);
  float k[U];
  bool near = false;
#pragma unroll
  for (int e = 0; e < U; e += 2) {
    const unsigned long long qa = mul2(pack2(y[e], y[e + 1]), r2);
    const unsigned long long r = sub2(add2(qa, m2), m2);
    const unsigned long long df = sub2(qa, r);
    near |= !(fabsf(lo2(df)) < kBand) || !(fabsf(hi2(df)) < kBand);
    k[e] = lo2(r);
    k[e + 1] = hi2(r);
  }
  if (near) {  // rare: the quotients themselves
#pragma unroll
    for (int e = 0; e < U; ++e) {
      const float r = rintf(__fdiv_rn(y[e], d));
      k[e] = r == r ? r : 0.0f;
    }
  }
  uint32_t out = 0;
#pragma unroll
  for (int e = 0; e < U; ++e)
    out |= (__float_as_uint(fminf(fmaxf(k[e], -8.0f), 7.0f) + (kMagic + 8.0f)) & 15u) << (4 * e);
  return out;
}

// Lane-group row shape of the bulk int8 and K8V4 appends: a row (one token
// and KV head, K and V) is held by a group of LPR consecutive lanes, lane j
// of the group holding the VPL consecutive dims j VPL .. j VPL + VPL - 1
// (64 contiguous bytes of fp32 at VPL 16), so a warp carries 32 / LPR rows
// at once.  Bulk appends take VPL = 16 (8 at HD 64): few shuffles per row;
// a few K8V4 rows (decode steps) take VPL = 4 (8 at HD 256): short chains.
template <int HD, int VPL_>
struct LaneRows {
  static constexpr int VPL = VPL_;                // values a lane holds (4, 8 or 16)
  static constexpr int LPR = HD / VPL;            // lanes of a row
  static constexpr int RPW = 32 / LPR;            // rows a warp holds
  static_assert(VPL % 4 == 0 && LPR <= 32 && LPR * VPL == HD, "K8V4 row shape");
};

// int8 codes of one row held by a lane group (LaneRows layout): the group
// maximum over the 64 / VPL lanes of each 64-dim group (bit patterns of |x|,
// as the int8 kernel), group_scale, codes4 (or the quotients for a
// non-finite group); dr < 0 stores nothing.
template <int HD, int VPL, int LPR>
__device__ __forceinline__ void q8_lanes(const float (&x)[VPL], long long dr, int j, int8_t* codes,
                                         __half* scales) {
  constexpr int NG = HD / kGroup;
  constexpr int LG = kGroup / VPL;  // lanes of a 64-dim group
  uint32_t mb = 0;
#pragma unroll
  for (int e = 0; e < VPL; ++e) mb = max(mb, __float_as_uint(x[e]) & 0x7fffffffu);
#pragma unroll
  for (int off = 1; off < LG; off <<= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, off));
  const float amax = __uint_as_float(mb);
  const __half sh = group_scale(amax);
  const float sf = __half2float(sh);
  uint32_t c[VPL / 4];
  if (amax <= 3.4028234663852886e38f) {
    const float rs = rcp_approx(sf);
#pragma unroll
    for (int q = 0; q < VPL / 4; ++q)
      c[q] = codes4(make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]), sf, rs);
  } else {
#pragma unroll
    for (int q = 0; q < VPL / 4; ++q)
      c[q] = exact_code(x[4 * q], sf) | (exact_code(x[4 * q + 1], sf) << 8) |
             (exact_code(x[4 * q + 2], sf) << 16) | (exact_code(x[4 * q + 3], sf) << 24);
  }
  if (dr >= 0) {
    int8_t* dst = codes + dr * HD + j * VPL;
    if constexpr (VPL == 16)
      *reinterpret_cast<uint4*>(dst) = make_uint4(c[0], c[1], c[VPL > 8 ? 2 : 0], c[VPL > 8 ? 3 : 0]);
    else if constexpr (VPL == 8)
      *reinterpret_cast<uint2*>(dst) = make_uint2(c[0], c[VPL > 4 ? 1 : 0]);
    else
      *reinterpret_cast<uint32_t*>(dst) = c[0];
    if (j % LG == 0) scales[dr * NG + (j * VPL) / kGroup] = sh;
  }
}

// Loads of one row into a lane group (zeros for rows past the end).
template <int HD, int VPL>
__device__ __forceinline__ void load_row_lanes(const float* src, long long row, bool live, int j,
                                               float (&x)[VPL]) {
#pragma unroll
  for (int q = 0; q < VPL / 4; ++q) {
    float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) v4 = __ldcs(reinterpret_cast<const float4*>(src + (size_t)row * HD + (size_t)j * VPL + 4 * q));
    x[4 * q] = v4.x;
    x[4 * q + 1] = v4.y;
    x[4 * q + 2] = v4.z;
    x[4 * q + 3] = v4.w;
  }
}

// int8 append of bulk batches (prefill, prompt chunks) with the lane-group
// row layout: K and V of a row each through q8_lanes.  Same arithmetic,
// hence the same bytes, as append_q8_kernel; about 1.3x its rate, since
// every lane keeps 128 contiguous bytes of K and V in flight.
template <int HD, int VPL_, int W>
__global__ void __launch_bounds__(W * 32) append_q8_rows_kernel(AppendArgs a) {
  using R = LaneRows<HD, VPL_>;
  constexpr int VPL = R::VPL, LPR = R::LPR, RPW = R::RPW;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31, j = lane & (LPR - 1);
  const long long rows = (long long)a.n_tok * a.n_kv;
  const bool rows32 = rows <= 0x7fffffffLL;
  const long long row0 = ((long long)blockIdx.x * W + (threadIdx.x >> 5)) * RPW;
  if (row0 >= rows) return;  // warp-uniform
  const long long row = row0 + lane / LPR;
  const bool live = row < rows;
  float xk[VPL], xv[VPL];
  load_row_lanes<HD, VPL>(a.k, row, live, j, xk);
  load_row_lanes<HD, VPL>(a.v, row, live, j, xv);
  const long long dr = live ? dest_row(a, row, rows32) : -1;
  q8_lanes<HD, VPL, LPR>(xk, dr, j, static_cast<int8_t*>(a.k_dst), a.ks_dst);
  q8_lanes<HD, VPL, LPR>(xv, dr, j, static_cast<int8_t*>(a.v_dst), a.vs_dst);
}

// K8V4 append (LaneRows layout; W warps a CTA).  K: int8 codes per 64-dim
// group, the int8 format's arithmetic (group maximum over the group's
// lanes, group_scale, codes4).  V: rotated (wht_group), then per block of
// 32 rotated dims the element of largest magnitude, the first one on ties
// (the block maximum of |y|, then the lowest dim holding it; NaN counts as
// 0 and a zero maximum gives m = +0, as the comparison-based definition
// does), d = fp16(m / -8), and two codes a byte.  Rows past the end carry
// zeros through every shuffle and store nothing.
template <int HD, int VPL_, int W>
__global__ void __launch_bounds__(W * 32) append_k8v4_kernel(AppendArgs a) {
  using R = LaneRows<HD, VPL_>;
  constexpr int VPL = R::VPL, LPR = R::LPR, RPW = R::RPW;
  constexpr int NB = HD / kQ4Block;
  constexpr int LB = kQ4Block / VPL;  // lanes of a 32-dim V block
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31, j = lane & (LPR - 1);
  const long long rows = (long long)a.n_tok * a.n_kv;
  const bool rows32 = rows <= 0x7fffffffLL;
  const long long row0 = ((long long)blockIdx.x * W + (threadIdx.x >> 5)) * RPW;
  if (row0 >= rows) return;  // warp-uniform; no block-level barrier follows
  const long long row = row0 + lane / LPR;
  const bool live = row < rows;

  float xk[VPL], xv[VPL];
  load_row_lanes<HD, VPL>(a.k, row, live, j, xk);
  load_row_lanes<HD, VPL>(a.v, row, live, j, xv);
  const long long dr = live ? dest_row(a, row, rows32) : -1;

  // ---- K: int8, one fp16 scale per 64 dims
  q8_lanes<HD, VPL, LPR>(xk, dr, j, static_cast<int8_t*>(a.k_dst), a.ks_dst);

  // ---- V: rotate, then 4-bit codes and one fp16 scale per 32 rotated dims
  wht_group<VPL, LPR>(xv, lane);
  {
    // the block's largest |y| (fmaxf drops NaN, so NaN counts as 0) ...
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < VPL; ++e) amax = fmaxf(amax, fabsf(xv[e]));
#pragma unroll
    for (int off = 1; off < LB; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    // ... and the first dim holding it: the lowest lane of the block with a
    // match (lanes hold ascending dims), then its lowest element (the
    // backward scan keeps the lowest)
    float mine = 0.f;
    bool found = false;
#pragma unroll
    for (int e = VPL - 1; e >= 0; --e)
      if (fabsf(xv[e]) == amax) {
        mine = xv[e];
        found = true;
      }
    const unsigned blk_lanes = ((1u << LB) - 1u) << (lane & ~(LB - 1));
    const unsigned hit = __ballot_sync(0xffffffffu, found) & blk_lanes;
    const int src = hit ? __ffs(hit) - 1 : lane;  // no match only if amax is 0 (all NaN)
    float m = __shfl_sync(0xffffffffu, mine, src);
    if (amax == 0.f) m = 0.0f;  // no nonzero element: m stays +0
    const __half dh = __float2half_rn(m * -0.125f);  // = m / -8, both correctly rounded
    const float d = __half2float(dh);
    uint32_t c[VPL / 4];  // 4 codes (16 bits) each; dims 2i low nibble, 2i + 1 high
#pragma unroll
    for (int q = 0; q < VPL / 4; ++q) {
      const float y4[4] = {xv[4 * q], xv[4 * q + 1], xv[4 * q + 2], xv[4 * q + 3]};
      c[q] = q4_codes<4>(y4, d);
    }
    if (dr >= 0) {
      uint8_t* dst = static_cast<uint8_t*>(a.v_dst) + dr * (HD / 2) + j * (VPL / 2);
      if constexpr (VPL == 16)
        *reinterpret_cast<uint2*>(dst) = make_uint2(c[0] | (c[1] << 16), c[VPL > 8 ? 2 : 0] | (c[VPL > 8 ? 3 : 0] << 16));
      else if constexpr (VPL == 8)
        *reinterpret_cast<uint32_t*>(dst) = c[0] | (c[VPL > 4 ? 1 : 0] << 16);
      else
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)c[0];
      if (j % LB == 0) a.vs_dst[dr * NB + (j * VPL) / kQ4Block] = dh;
    }
  }
}

template <typename Kernel>
cudaError_t launch_grid(Kernel kern, long long blocks, int threads, const AppendArgs& a,
                        cudaStream_t s) {
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// Bulk appends (prefill, prompt chunks) keep several 16-byte loads in
// flight per thread; a few tokens (decode steps) use small CTAs, so the work
// spreads over more SMs and no thread runs a long serial chain.
template <int HD>
cudaError_t launch_f16(const AppendArgs& a, cudaStream_t s) {
  const long long chunks = (long long)a.n_tok * a.n_kv * (HD / 4);
  if (chunks < (1LL << 16)) return launch_grid(append_f16_kernel<HD, 1, 2>, (chunks + 63) / 64, 64, a, s);
  return launch_grid(append_f16_kernel<HD, 4, 8>, (chunks + 1023) / 1024, 256, a, s);
}

template <int HD>
cudaError_t launch_q8(const AppendArgs& a, cudaStream_t s) {
  const long long groups = (long long)a.n_tok * a.n_kv * (HD / kGroup);
  if (groups < (1LL << 12))
    return launch_grid(append_q8_kernel<HD, 1, 2, true>, (groups + 7) / 8, 64, a, s);
  constexpr int VB = HD >= 128 ? 16 : 8;
  constexpr int RB = LaneRows<HD, VB>::RPW;
  const long long rows = (long long)a.n_tok * a.n_kv;
  return launch_grid(append_q8_rows_kernel<HD, VB, 8>, (rows + 8 * RB - 1) / (8 * RB), 256, a, s);
}

// Few rows (decode steps): short per-lane chains (VPL 4, 8 at HD 256) in
// CTAs of 4 warps; bulk: VPL 16 (8 at HD 64) in CTAs of 8 warps.
template <int HD>
cudaError_t launch_k8v4(const AppendArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.n_tok * a.n_kv;
  constexpr int VS = HD == 256 ? 8 : 4, VB = HD >= 128 ? 16 : 8;
  constexpr int RS = LaneRows<HD, VS>::RPW, RB = LaneRows<HD, VB>::RPW;
  if (rows < 4096)
    return launch_grid(append_k8v4_kernel<HD, VS, 4>, (rows + 4 * RS - 1) / (4 * RS), 128, a, s);
  return launch_grid(append_k8v4_kernel<HD, VB, 8>, (rows + 8 * RB - 1) / (8 * RB), 256, a, s);
}

template <int HD>
cudaError_t launch_hd(int fmt, const AppendArgs& a, cudaStream_t s) {
  if (fmt == KVQ_F16) return launch_f16<HD>(a, s);
  if (fmt == KVQ_Q8) return launch_q8<HD>(a, s);
  if (fmt == KVQ_K8V4) return launch_k8v4<HD>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_append(int fmt, int hd, const AppendArgs& a, cudaStream_t s) {
  switch (hd) {
    case 64: return launch_hd<64>(fmt, a, s);
    case 128: return launch_hd<128>(fmt, a, s);
    case 256: return launch_hd<256>(fmt, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq

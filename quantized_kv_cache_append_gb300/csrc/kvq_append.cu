// kvq_append.cu -- quantize-on-write of new K/V rows into the paged pool.
//
// #3084 qwen35: FP16 K/V cache by default, int8 with --kv-q8, "What changed":
// under --kv-q8 a row is written as scale = fp16(max|x| / 127) per 64 dims and
// code = clamp(rint(x / scale), -127, 127); the FP16 cache stores fp16(x).
// The same section notes that the group maximum needs every thread to reach
// a barrier before the stores.  Here one warp owns one row (one cell, one KV
// head, K or V), so the group maximum is a warp-shuffle butterfly: no
// __syncthreads exists in this kernel and no early return can skip one.
//
// Bit-exactness: max|x| is exact; a / 127.0f and x / s are IEEE fp32
// divisions (the library is built without fast-math, so '/' is div.rn.f32);
// __float2half_rn rounds to nearest even with subnormals; __float2int_rn
// rounds half to even and saturates, so clamping afterwards equals clamping
// the rounded value.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

// Butterfly max over the `kLanes` lanes that share one 64-dim group.
template <int kLanes>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int off = kLanes / 2; off >= 1; off >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ int quantize_one(float x, float sf) {
  if (sf == 0.0f) return 0;
  int c = __float2int_rn(x / sf);
  return max(-127, min(127, c));
}

// One warp per row.  A row of HD fp32 values is read as CHUNKS chunks of 32
// lanes x VEC consecutive floats; lane l holds dims [chunk*32*VEC + l*VEC,
// + VEC), so each 64-dim group is 64/VEC consecutive lanes.
template <int FMT, int HD>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  constexpr int VEC = HD >= 128 ? 4 : 2;
  constexpr int CHUNK = 32 * VEC;
  constexpr int CHUNKS = HD / CHUNK;
  constexpr int LANES_PER_GROUP = kGroup / VEC;
  constexpr int NG = HD / kGroup;

  // Launched as a programmatic dependent: wait for the previous kernel's
  // writes (k, v, positions may come from it), then let the next kernel's
  // launch begin.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const long long n_rows = (long long)a.n_tok * a.n_kv * 2;
  if (row >= n_rows) return;  // warp-uniform; the kernel has no block barrier

  const int which = (int)(row & 1);  // 0 = K, 1 = V
  const long long tk = row >> 1;     // token * n_kv + kvh
  const int tok = (int)(tk / a.n_kv);
  const int kvh = (int)(tk - (long long)tok * a.n_kv);

  const int seq = __ldg(a.tok_seq + tok);
  const int pos = __ldg(a.tok_pos + tok);
  const int bs = 1 << a.bs_log2;
  if (seq < 0 || seq >= a.n_seq || pos < 0 || (pos >> a.bs_log2) >= a.max_blocks) return;
  const int blk = __ldg(a.block_table + (size_t)seq * a.max_blocks + (pos >> a.bs_log2));
  if (blk < 0 || blk >= a.n_blocks) return;  // precondition broken: write nothing
  const size_t dst_row = ((size_t)blk * a.n_kv + kvh) * bs + (pos & (bs - 1));

  const float* src = (which ? a.v : a.k) + (size_t)tk * HD;

  float x[CHUNKS][VEC];
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    const float* p = src + c * CHUNK + lane * VEC;
    if constexpr (VEC == 4) {
      const float4 t = __ldg(reinterpret_cast<const float4*>(p));
      x[c][0] = t.x; x[c][1] = t.y; x[c][2] = t.z; x[c][3] = t.w;
    } else {
      const float2 t = __ldg(reinterpret_cast<const float2*>(p));
      x[c][0] = t.x; x[c][1] = t.y;
    }
  }

  if constexpr (FMT == KVQ_F16) {
    __half* dst = static_cast<__half*>(which ? a.v_dst : a.k_dst) + dst_row * HD;
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
      __half h[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) h[e] = __float2half_rn(x[c][e]);
      __half* p = dst + c * CHUNK + lane * VEC;
      if constexpr (VEC == 4) {
        uint2 u;
        u.x = (uint32_t)__half_as_ushort(h[0]) | ((uint32_t)__half_as_ushort(h[1]) << 16);
        u.y = (uint32_t)__half_as_ushort(h[2]) | ((uint32_t)__half_as_ushort(h[3]) << 16);
        *reinterpret_cast<uint2*>(p) = u;
      } else {
        const uint32_t u =
            (uint32_t)__half_as_ushort(h[0]) | ((uint32_t)__half_as_ushort(h[1]) << 16);
        *reinterpret_cast<uint32_t*>(p) = u;
      }
    }
  } else {
    int8_t* dst = static_cast<int8_t*>(which ? a.v_dst : a.k_dst) + dst_row * HD;
    __half* sdst = (which ? a.vs_dst : a.ks_dst) + dst_row * NG;
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < VEC; ++e) amax = fmaxf(amax, fabsf(x[c][e]));
      amax = group_max<LANES_PER_GROUP>(amax);
      const __half s = __float2half_rn(amax / 127.0f);
      const float sf = __half2float(s);
      uint32_t packed = 0;
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        packed |= ((uint32_t)(quantize_one(x[c][e], sf) & 0xff)) << (8 * e);
      int8_t* p = dst + c * CHUNK + lane * VEC;
      if constexpr (VEC == 4)
        *reinterpret_cast<uint32_t*>(p) = packed;
      else
        *reinterpret_cast<uint16_t*>(p) = (uint16_t)packed;
      if ((lane % LANES_PER_GROUP) == 0) {
        const int g = (c * CHUNK + lane * VEC) / kGroup;
        sdst[g] = s;
      }
    }
  }
}

template <int FMT>
cudaError_t launch_fmt(int hd, const AppendArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.n_tok * a.n_kv * 2;
  const int warps_per_block = 8;
  const long long blocks = (rows + warps_per_block - 1) / warps_per_block;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(32 * warps_per_block);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (hd) {
    case 64: return cudaLaunchKernelEx(&cfg, append_kernel<FMT, 64>, a);
    case 128: return cudaLaunchKernelEx(&cfg, append_kernel<FMT, 128>, a);
    case 256: return cudaLaunchKernelEx(&cfg, append_kernel<FMT, 256>, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_append(int fmt, int hd, const AppendArgs& a, cudaStream_t s) {
  return fmt == KVQ_F16 ? launch_fmt<KVQ_F16>(hd, a, s) : launch_fmt<KVQ_Q8>(hd, a, s);
}

}  // namespace kvq

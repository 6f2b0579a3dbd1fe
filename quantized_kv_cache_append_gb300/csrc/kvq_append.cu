// kvq_append.cu -- quantize-on-write of new K/V rows into the paged pool.
//
// #3084 qwen35: FP16 K/V cache by default, int8 with --kv-q8, "What changed":
// under --kv-q8 a row is written as scale = fp16(max|x| / 127) per 64 dims and
// code = clamp(rint(x / scale), -127, 127); the FP16 cache stores fp16(x).
// The same section notes that the group maximum needs every thread to reach
// a barrier before the stores.  Here one half-warp owns one 64-dim group, so
// the group maximum is a warp-shuffle butterfly that every lane executes: no
// __syncthreads exists in this kernel and no early return can skip one.
//
// Bit-exactness: max|x| is exact; a / 127.0f is an IEEE fp32 division (the
// library is built without fast-math, so '/' is div.rn.f32); x / s is
// replaced by a reciprocal multiply only where that provably rounds to the
// same integer (quantize_one); __float2half_rn rounds to nearest even with
// subnormals; rintf rounds half to even, so clamping afterwards equals
// clamping the rounded value.
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

// code = clamp(rint(x / sf), -127, 127) with x / sf the IEEE fp32 quotient.
// y = x * (1 / sf) is within about 2^-22 |x / sf| of the real quotient (both
// roundings together), and |x / sf| stays below 256, so wherever y lies
// more than 2.5e-4 away from a half-integer, the real quotient, its fp32
// rounding and y all round to the same integer.  Only inside that band is
// the quotient itself computed (a few elements in ten thousand), so ties
// and near-ties resolve exactly as the division defines them.
__device__ __forceinline__ int quantize_one(float x, float sf, float rs) {
  if (sf == 0.0f) return 0;
  const float y = x * rs;
  float n = rintf(y);
  if (fabsf(fabsf(y - n) - 0.5f) < 2.5e-4f) n = rintf(x / sf);
  const int c = __float2int_rn(n);  // NaN (out-of-domain input) gives 0
  return max(-127, min(127, c));
}

// The K and V inputs are flat arrays of n_tok * n_kv * HD floats, read as
// 16-byte chunks; a 64-dim group is 16 consecutive chunks, so one half-warp
// owns one group and finds its maximum with a 4-step butterfly.  Each thread
// handles U chunk positions of K and the same positions of V (2U loads in
// flight before the first use), warp j covering chunks [32 U j, 32 U (j+1));
// a CTA has W warps.
// The destination of a row comes from the token's sequence, position and
// block-table entry; those small loads are issued beside the data loads.
template <int HD, int U, int W>
struct AppendShape {
  static constexpr int CPR = HD / 4;   // 16-byte chunks per row
  static constexpr int WARPS = W;      // warps per CTA
  static constexpr long long CHUNKS_PER_CTA = 32LL * U * WARPS;
};

template <int FMT, int HD, int U, int W>
__global__ void __launch_bounds__(W * 32) append_kernel(AppendArgs a) {
  using S = AppendShape<HD, U, W>;
  constexpr int NG = HD / kGroup;

  // Launched as a programmatic dependent: wait for the previous kernel's
  // writes (k, v, positions may come from it), then let the next kernel's
  // launch begin.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long n_chunks = (long long)a.n_tok * a.n_kv * S::CPR;  // a multiple of 16
  const long long base = (long long)blockIdx.x * S::CHUNKS_PER_CTA + (threadIdx.x >> 5) * 32LL * U;
  const float4* k4 = reinterpret_cast<const float4*>(a.k);
  const float4* v4 = reinterpret_cast<const float4*>(a.v);

  float4 xk[U], xv[U];
  long long dst_row[U];
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const long long f = base + 32LL * j + lane;
    xk[j] = xv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    dst_row[j] = -1;
    if (f < n_chunks) {
      xk[j] = __ldcs(k4 + f);
      xv[j] = __ldcs(v4 + f);
    }
  }
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const long long f = base + 32LL * j + lane;
    if (f < n_chunks) {
      const long long row = f / S::CPR;                 // token * n_kv + kvh
      const int tok = (int)(row / a.n_kv);
      const int kvh = (int)(row - (long long)tok * a.n_kv);
      const int seq = __ldg(a.tok_seq + tok);
      const int pos = __ldg(a.tok_pos + tok);
      if (seq >= 0 && seq < a.n_seq && pos >= 0 && (pos >> a.bs_log2) < a.max_blocks) {
        const int blk = __ldg(a.block_table + (size_t)seq * a.max_blocks + (pos >> a.bs_log2));
        if (blk >= 0 && blk < a.n_blocks)  // precondition broken: write nothing
          dst_row[j] = ((long long)blk * a.n_kv + kvh) * (1LL << a.bs_log2) +
                       (pos & ((1 << a.bs_log2) - 1));
      }
    }
  }

#pragma unroll
  for (int j = 0; j < U; ++j) {
    const long long f = base + 32LL * j + lane;
    const int d = (int)(f % S::CPR) * 4;                // first dim of this chunk
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const float4 x = which ? xv[j] : xk[j];
      if constexpr (FMT == KVQ_F16) {
        if (dst_row[j] >= 0) {
          __half* dst = static_cast<__half*>(which ? a.v_dst : a.k_dst) + dst_row[j] * HD + d;
          uint2 u;
          u.x = (uint32_t)__half_as_ushort(__float2half_rn(x.x)) |
                ((uint32_t)__half_as_ushort(__float2half_rn(x.y)) << 16);
          u.y = (uint32_t)__half_as_ushort(__float2half_rn(x.z)) |
                ((uint32_t)__half_as_ushort(__float2half_rn(x.w)) << 16);
          *reinterpret_cast<uint2*>(dst) = u;
        }
      } else {
        // every lane takes part in the butterfly (out-of-range half-warps
        // carry zeros and store nothing)
        float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
        amax = group_max<16>(amax);
        const __half sh = __float2half_rn(amax / 127.0f);
        const float sf = __half2float(sh);
        const float rs = 1.0f / sf;
        if (dst_row[j] >= 0) {
          const uint32_t packed = ((uint32_t)(quantize_one(x.x, sf, rs) & 0xff)) |
                                  ((uint32_t)(quantize_one(x.y, sf, rs) & 0xff) << 8) |
                                  ((uint32_t)(quantize_one(x.z, sf, rs) & 0xff) << 16) |
                                  ((uint32_t)(quantize_one(x.w, sf, rs) & 0xff) << 24);
          int8_t* dst = static_cast<int8_t*>(which ? a.v_dst : a.k_dst) + dst_row[j] * HD + d;
          *reinterpret_cast<uint32_t*>(dst) = packed;
          if ((lane & 15) == 0)
            (which ? a.vs_dst : a.ks_dst)[dst_row[j] * NG + d / kGroup] = sh;
        }
      }
    }
  }
}

template <int FMT, int HD, int U, int W>
cudaError_t launch_shape(const AppendArgs& a, cudaStream_t s) {
  using S = AppendShape<HD, U, W>;
  const long long chunks = (long long)a.n_tok * a.n_kv * S::CPR;
  const long long blocks = (chunks + S::CHUNKS_PER_CTA - 1) / S::CHUNKS_PER_CTA;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(32 * S::WARPS);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_kernel<FMT, HD, U, W>, a);
}

// Bulk appends (prefill, prompt chunks) keep 8 chunks of 16 bytes in flight
// per thread; a few tokens (decode steps) take one chunk of K and one of V
// per thread in small CTAs, so the work spreads over more SMs and no thread
// runs a long serial chain of group maxima.
template <int FMT, int HD>
cudaError_t launch_hd(const AppendArgs& a, cudaStream_t s) {
  const long long chunks = (long long)a.n_tok * a.n_kv * (HD / 4);
  if (chunks < (1LL << 16)) return launch_shape<FMT, HD, 1, 2>(a, s);
  return launch_shape<FMT, HD, 4, 8>(a, s);
}

template <int FMT>
cudaError_t launch_fmt(int hd, const AppendArgs& a, cudaStream_t s) {
  switch (hd) {
    case 64: return launch_hd<FMT, 64>(a, s);
    case 128: return launch_hd<FMT, 128>(a, s);
    case 256: return launch_hd<FMT, 256>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_append(int fmt, int hd, const AppendArgs& a, cudaStream_t s) {
  return fmt == KVQ_F16 ? launch_fmt<KVQ_F16>(hd, a, s) : launch_fmt<KVQ_Q8>(hd, a, s);
}

}  // namespace kvq

// kvq_decode.cu -- split-K GQA decode attention over the paged K/V pool.
//
// #3084 qwen35: FP16 K/V cache by default, int8 with --kv-q8, "What changed"
// and "Extra Notes": the decode of the next token reads the cache through a
// split-K partial kernel (k_attn_part, templated on the cache format) whose
// partial results are merged afterwards.  Here:
//
//   partial kernel  one CTA per (split, KV head, sequence).  It streams the
//                   split's cells once, dequantizes K and V in registers
//                   (k = code * scale, exact), and runs the G * W query rows
//                   of that KV head (GQA heads sharing one K/V read) with an
//                   online softmax in the log2 domain.  It writes an
//                   unnormalised partial output o_j and (m_j, l_j) per row.
//   combine kernel  one CTA per output row: M = max_j m_j,
//                   out = sum_j 2^(m_j - M) o_j / sum_j 2^(m_j - M) l_j.
//                   It is launched as a programmatic dependent of the
//                   partial kernel and waits on griddepcontrol before it
//                   reads the partials.
//
// Rows r = w * G + g: query token w of the window, head kvh * G + g.  Token
// w sees cells [0, L - W + w].  A row with no visible cell outputs zeros.
//
// K8V4 (#711 kv: --kv k8v4 streams with --kv-resident, "What"): K is read
// as int8; V as (nibble - 8) * d in the rotated basis, the CTA's merged
// partial is rotated back (Walsh-Hadamard, divided by HD) before it is
// written, and the combine, being linear in the partials, is unchanged.
#include <math.h>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kWarps = 4;
constexpr int kTile = 32;                  // cells per warp tile (lane = cell)
constexpr int kCellTile = kWarps * kTile;  // split sizes are multiples of this
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
  return v;
}

// ctx_lens[b] limited to the cells the block table row and the split plan
// can address (a broken precondition must not read past the table).
__device__ __forceinline__ int clamp_len(int L, const DecodeArgs& a) {
  const long long cap_table = (long long)a.max_blocks << a.pool.bs_log2;
  const long long cap_plan = (long long)a.nsplit * a.split_cells;
  long long cap = cap_table < cap_plan ? cap_table : cap_plan;
  return L < 0 ? 0 : (int)((long long)L < cap ? L : cap);
}

// Element e (0..3) of four packed int8 codes, or (0..1) of two packed fp16.
__device__ __forceinline__ float code_i8(uint32_t w, int e) {
  return (float)(int8_t)(w >> (8 * e));
}
__device__ __forceinline__ float code_f16(uint32_t w, int e) {
  return __half2float(__ushort_as_half((unsigned short)(w >> (16 * e))));
}

template <int FMT, int HD, int RP>
__global__ void __launch_bounds__(kWarps * 32) decode_partial(DecodeArgs a) {
  constexpr int E = HD / 32;                // dims per lane in the P.V phase
  constexpr int NG = HD / kGroup;
  constexpr int ESZ = FMT == KVQ_F16 ? 2 : 1;  // K (and F16 / int8 V) element bytes
  constexpr int EPW = 4 / ESZ;              // elements per 32-bit word
  constexpr bool V4 = FMT == KVQ_K8V4;
  constexpr float kNegInf = -INFINITY;

  __shared__ __align__(16) float s_q[HD][RP];           // q * sm_scale * log2(e), [d][r]
  __shared__ __align__(16) float s_p[kWarps][kTile][RP];
  __shared__ float s_m[kWarps][RP];
  __shared__ float s_l[kWarps][RP];
  __shared__ __align__(16) float s_o[RP][HD];

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = clamp_len(__ldg(a.ctx_lens + b), a);
  const int c_begin = split * a.split_cells;
  if (c_begin >= L) return;  // empty split: the whole CTA leaves before any barrier
  const int c_end = min(L, c_begin + a.split_cells);
  const int bs_log2 = a.pool.bs_log2;
  const int bs = 1 << bs_log2;
  const int32_t* bt = a.block_table + (size_t)b * a.max_blocks;

  for (int i = threadIdx.x; i < HD * RP; i += blockDim.x) {
    const int r = i / HD, d = i - r * HD;
    float val = 0.0f;
    if (r < a.R) {
      const int w = r / a.G, g = r - w * a.G;
      val = a.q[(((size_t)b * a.W + w) * a.n_q + (size_t)kvh * a.G + g) * HD + d] * a.qscale;
    }
    s_q[d][r] = val;
  }
  __syncthreads();

  float m[RP], l[RP], o[RP][E];
#pragma unroll
  for (int r = 0; r < RP; ++r) {
    m[r] = kNegInf;
    l[r] = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[r][e] = 0.0f;
  }

  for (int tb = c_begin + warp * kTile; tb < c_end; tb += kWarps * kTile) {
    const int c = tb + lane;
    const bool valid = c < c_end;
    int row = -1;
    if (valid) {
      const int blk = __ldg(bt + (c >> bs_log2));
      if (blk >= 0 && blk < a.pool.n_blocks) row = (blk * a.pool.n_kv + kvh) * bs + (c & (bs - 1));
    }

    // ---- q . k for this lane's cell, all RP rows
    float z[RP];
#pragma unroll
    for (int r = 0; r < RP; ++r) z[r] = 0.0f;
    if (row >= 0) {
      const uint8_t* kp = static_cast<const uint8_t*>(a.pool.k) + (size_t)row * HD * ESZ;
      uint32_t sc_bits[NG];
      if constexpr (FMT != KVQ_F16) {
        const unsigned short* ks =
            reinterpret_cast<const unsigned short*>(a.pool.ks) + (size_t)row * NG;
#pragma unroll
        for (int g = 0; g < NG; ++g) sc_bits[g] = __ldg(ks + g);
      }
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        float part[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) part[r] = 0.0f;
#pragma unroll
        for (int ch = 0; ch < kGroup * ESZ / 16; ++ch) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(kp + g * kGroup * ESZ + ch * 16));
          const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
            for (int e = 0; e < EPW; ++e) {
              const int d = g * kGroup + ch * (16 / ESZ) + wi * EPW + e;
              const float x = FMT != KVQ_F16 ? code_i8(words[wi], e) : code_f16(words[wi], e);
#pragma unroll
              for (int r4 = 0; r4 < RP / 4; ++r4) {
                const float4 qv = *reinterpret_cast<const float4*>(&s_q[d][r4 * 4]);
                part[r4 * 4 + 0] = fmaf(qv.x, x, part[r4 * 4 + 0]);
                part[r4 * 4 + 1] = fmaf(qv.y, x, part[r4 * 4 + 1]);
                part[r4 * 4 + 2] = fmaf(qv.z, x, part[r4 * 4 + 2]);
                part[r4 * 4 + 3] = fmaf(qv.w, x, part[r4 * 4 + 3]);
              }
            }
          }
        }
        if constexpr (FMT != KVQ_F16) {
          const float sf = __half2float(__ushort_as_half((unsigned short)sc_bits[g]));
#pragma unroll
          for (int r = 0; r < RP; ++r) z[r] = fmaf(part[r], sf, z[r]);
        } else {
#pragma unroll
          for (int r = 0; r < RP; ++r) z[r] += part[r];
        }
      }
    }

    // ---- causal limit and online softmax (log2 domain)
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      const int last = L - a.W + r / a.G;
      if (!valid || c > last || r >= a.R) z[r] = kNegInf;
      const float mn = fmaxf(m[r], warp_max(z[r]));
      const float alpha = mn == kNegInf ? 1.0f : exp2f(m[r] - mn);
      const float p = mn == kNegInf ? 0.0f : exp2f(z[r] - mn);
      l[r] = fmaf(l[r], alpha, p);
      m[r] = mn;
#pragma unroll
      for (int e = 0; e < E; ++e) o[r][e] *= alpha;
      s_p[warp][lane][r] = p;
    }
    __syncwarp();

    // ---- p . v: lane owns dims [lane * E, lane * E + E)
    const int n_here = min(kTile, c_end - tb);
    for (int cc = 0; cc < n_here; ++cc) {
      const int rowc = __shfl_sync(kFull, row, cc);
      if (rowc < 0) continue;
      float pr[RP];
#pragma unroll
      for (int r4 = 0; r4 < RP / 4; ++r4) {
        const float4 pv = *reinterpret_cast<const float4*>(&s_p[warp][cc][r4 * 4]);
        pr[r4 * 4 + 0] = pv.x;
        pr[r4 * 4 + 1] = pv.y;
        pr[r4 * 4 + 2] = pv.z;
        pr[r4 * 4 + 3] = pv.w;
      }
      if constexpr (V4) {
        // lane's E dims: E / 2 bytes of nibbles, one scale (E <= 32)
        const uint8_t* vp = static_cast<const uint8_t*>(a.pool.v) + (size_t)rowc * (HD / 2) + lane * E / 2;
        const float sv = __half2float(__ldg(a.pool.vs + (size_t)rowc * (HD / kQ4Block) + (lane * E) / kQ4Block));
#pragma unroll
        for (int r = 0; r < RP; ++r) pr[r] *= sv;
        uint32_t bits;
        if constexpr (E == 2) bits = __ldg(vp);
        else if constexpr (E == 4) bits = __ldg(reinterpret_cast<const unsigned short*>(vp));
        else bits = __ldg(reinterpret_cast<const uint32_t*>(vp));
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float x = (float)((int)((bits >> (4 * e)) & 15u) - 8);
#pragma unroll
          for (int r = 0; r < RP; ++r) o[r][e] = fmaf(pr[r], x, o[r][e]);
        }
        continue;
      }
      const uint8_t* vp =
          static_cast<const uint8_t*>(a.pool.v) + ((size_t)rowc * HD + lane * E) * ESZ;
      if constexpr (FMT == KVQ_Q8) {
        const unsigned short sb = __ldg(reinterpret_cast<const unsigned short*>(a.pool.vs) +
                                        (size_t)rowc * NG + (lane * E) / kGroup);
        const float sv = __half2float(__ushort_as_half(sb));
#pragma unroll
        for (int r = 0; r < RP; ++r) pr[r] *= sv;
      }
      constexpr int VBYTES = E * ESZ;  // 2, 4, 8 or 16
      uint32_t words[(VBYTES + 3) / 4];
      if constexpr (VBYTES == 2) {
        words[0] = __ldg(reinterpret_cast<const unsigned short*>(vp));
      } else if constexpr (VBYTES == 4) {
        words[0] = __ldg(reinterpret_cast<const uint32_t*>(vp));
      } else if constexpr (VBYTES == 8) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(vp));
        words[0] = u.x;
        words[1] = u.y;
      } else {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(vp));
        words[0] = u.x;
        words[1] = u.y;
        words[2] = u.z;
        words[3] = u.w;
      }
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float x = FMT == KVQ_Q8 ? code_i8(words[e / EPW], e % EPW)
                                      : code_f16(words[e / EPW], e % EPW);
#pragma unroll
        for (int r = 0; r < RP; ++r) o[r][e] = fmaf(pr[r], x, o[r][e]);
      }
    }
    __syncwarp();
  }

  // ---- merge the warps of this CTA
#pragma unroll
  for (int r = 0; r < RP; ++r) l[r] = warp_sum(l[r]);
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      s_m[warp][r] = m[r];
      s_l[warp][r] = l[r];
    }
  }
  __syncthreads();
  float wgt[RP];
#pragma unroll
  for (int r = 0; r < RP; ++r) {
    float M = s_m[0][r];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_m[w][r]);
    wgt[r] = (M == kNegInf || m[r] == kNegInf) ? 0.0f : exp2f(m[r] - M);
  }
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (warp == w) {
#pragma unroll
      for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float prev = w == 0 ? 0.0f : s_o[r][lane * E + e];
          s_o[r][lane * E + e] = fmaf(wgt[r], o[r][e], prev);
        }
    }
    __syncthreads();
  }

  const size_t base = (((size_t)b * a.pool.n_kv + kvh) * a.nsplit + split) * a.R;
  if constexpr (V4) {
    // rotate each merged row back: one warp per row
    constexpr int U = HD >= 128 ? 4 : 2, NI = HD / (32 * U);
    for (int r = warp; r < a.R; r += kWarps) {
      float x[NI][U];
#pragma unroll
      for (int i = 0; i < NI; ++i)
#pragma unroll
        for (int e = 0; e < U; ++e) x[i][e] = s_o[r][e + U * lane + 32 * U * i];
      wht_warp<U, NI>(x, lane);
#pragma unroll
      for (int i = 0; i < NI; ++i)
#pragma unroll
        for (int e = 0; e < U; ++e)
          a.ws_o[(base + r) * HD + e + U * lane + 32 * U * i] = x[i][e] * (1.0f / HD);
    }
  } else {
    for (int i = threadIdx.x; i < a.R * HD; i += blockDim.x) {
      const int r = i / HD, d = i - r * HD;
      a.ws_o[(base + r) * HD + d] = s_o[r][d];
    }
  }
  if (threadIdx.x < a.R) {
    const int r = threadIdx.x;
    float M = s_m[0][r];
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_m[w][r]);
    float lsum = 0.0f;
    for (int w = 0; w < kWarps; ++w)
      if (s_m[w][r] != kNegInf) lsum = fmaf(s_l[w][r], exp2f(s_m[w][r] - M), lsum);
    a.ws_ml[(base + r) * 2 + 0] = M;
    a.ws_ml[(base + r) * 2 + 1] = lsum;
  }
  // Let the combine grid get scheduled; it still waits for this grid to
  // complete (griddepcontrol.wait) before it reads any partial.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One CTA per output row (sequence, KV head, row r).  Threads are
// (j-slice, float4 of dims); slices are reduced through shared memory.
template <int HD>
__global__ void __launch_bounds__(256) decode_combine(DecodeArgs a) {
  constexpr int TPR = HD / 4;     // threads covering one row vector
  constexpr int JS = 256 / TPR;   // split slices
  constexpr float kNegInf = -INFINITY;
  __shared__ float s_red[256];
  __shared__ __align__(16) float4 s_acc[JS][TPR];
  __shared__ float s_lsum[JS];

  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int t = threadIdx.x;
  const int r = blockIdx.x % a.R;
  const int bk = blockIdx.x / a.R;
  const int kvh = bk % a.pool.n_kv;
  const int b = bk / a.pool.n_kv;
  const int L = clamp_len(__ldg(a.ctx_lens + b), a);
  const int ns = L <= 0 ? 0 : min(a.nsplit, (L + a.split_cells - 1) / a.split_cells);
  const int w = r / a.G, g = r - (r / a.G) * a.G;
  float* dst = a.out + (((size_t)b * a.W + w) * a.n_q + (size_t)kvh * a.G + g) * HD;
  const size_t base = ((size_t)b * a.pool.n_kv + kvh) * a.nsplit;

  // A partial whose producer lost an mbarrier wait carries m = NaN: the
  // row's output becomes NaN instead of a silently wrong value.
  float mx = kNegInf;
  int lost = 0;
  for (int j = t; j < ns; j += 256) {
    const float mj = __ldcg(a.ws_ml + ((base + j) * a.R + r) * 2);
    lost |= mj != mj;
    mx = fmaxf(mx, mj);
  }
  s_red[t] = mx;
  lost = __syncthreads_or(lost);
  for (int s = 128; s >= 1; s >>= 1) {
    if (t < s) s_red[t] = fmaxf(s_red[t], s_red[t + s]);
    __syncthreads();
  }
  const float M = s_red[0];
  if (lost) {
    if (t < TPR) {
      const float nan = __int_as_float(0x7fc00000);
      *reinterpret_cast<float4*>(dst + t * 4) = make_float4(nan, nan, nan, nan);
    }
    return;
  }

  const int d4 = (t % TPR) * 4, js = t / TPR;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.0f;
  if (M != kNegInf) {
    for (int j = js; j < ns; j += JS) {
      const size_t rj = (base + j) * a.R + r;
      const float mj = __ldcg(a.ws_ml + rj * 2 + 0);
      if (mj == kNegInf) continue;
      const float wj = exp2f(mj - M);
      lsum = fmaf(wj, __ldcg(a.ws_ml + rj * 2 + 1), lsum);
      const float4 oj = __ldcg(reinterpret_cast<const float4*>(a.ws_o + rj * HD + d4));
      acc.x = fmaf(wj, oj.x, acc.x);
      acc.y = fmaf(wj, oj.y, acc.y);
      acc.z = fmaf(wj, oj.z, acc.z);
      acc.w = fmaf(wj, oj.w, acc.w);
    }
  }
  s_acc[js][t % TPR] = acc;
  if (t % TPR == 0) s_lsum[js] = lsum;
  __syncthreads();
  if (t < TPR) {
    float4 sum = s_acc[0][t];
    float lt = s_lsum[0];
    for (int s = 1; s < JS; ++s) {
      const float4 v = s_acc[s][t];
      sum.x += v.x;
      sum.y += v.y;
      sum.z += v.z;
      sum.w += v.w;
      lt += s_lsum[s];
    }
    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != kNegInf && lt > 0.0f) {
      const float inv = 1.0f / lt;
      res = make_float4(sum.x * inv, sum.y * inv, sum.z * inv, sum.w * inv);
    }
    *reinterpret_cast<float4*>(dst + t * 4) = res;
  }
}

template <int FMT, int HD, int RP>
cudaError_t launch_partial(const DecodePlan& p, const DecodeArgs& a, cudaStream_t s) {
  const dim3 grid(p.nsplit, a.pool.n_kv, a.n_seq);
  decode_partial<FMT, HD, RP><<<grid, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

template <int FMT, int HD>
cudaError_t launch_rows(const DecodePlan& p, const DecodeArgs& a, cudaStream_t s) {
  constexpr int E = HD / 32;
  switch (p.rows_pad) {
    case 4: return launch_partial<FMT, HD, 4>(p, a, s);
    case 8: return launch_partial<FMT, HD, 8>(p, a, s);
    case 16:
      if constexpr (16 * E <= 64) return launch_partial<FMT, HD, 16>(p, a, s);
      break;
    case 32:
      if constexpr (32 * E <= 64) return launch_partial<FMT, HD, 32>(p, a, s);
      break;
  }
  return cudaErrorInvalidValue;
}

template <int HD>
cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_seq * a.pool.n_kv * a.R);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine<HD>, a);
}

}  // namespace

int decode_cell_tile() { return kCellTile; }

int decode_rows_pad(int hd, int rows) {
  (void)hd;
  int rp = 4;
  while (rp < rows) rp *= 2;
  return rp;
}

bool decode_supported(int fmt, int hd, int rows) {
  if (fmt != KVQ_F16 && fmt != KVQ_Q8 && fmt != KVQ_K8V4) return false;
  if (hd != 64 && hd != 128 && hd != 256) return false;
  if (mma_decode_supported(fmt, hd, rows)) return true;
  const int rp = decode_rows_pad(hd, rows);
  return rows >= 1 && rp <= 32 && rp * (hd / 32) <= 64;
}

cudaError_t launch_decode(int fmt, int hd, const DecodePlan& plan, const DecodeArgs& a,
                          cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidValue;
  if (plan.use_mma) {
    // the tensor-core partial kernel and its combine
    return launch_decode_mma_partial(fmt, hd, plan, a, s);
  } else if (fmt == KVQ_F16) {
    if (hd == 64) e = launch_rows<KVQ_F16, 64>(plan, a, s);
    else if (hd == 128) e = launch_rows<KVQ_F16, 128>(plan, a, s);
    else if (hd == 256) e = launch_rows<KVQ_F16, 256>(plan, a, s);
  } else if (fmt == KVQ_Q8) {
    if (hd == 64) e = launch_rows<KVQ_Q8, 64>(plan, a, s);
    else if (hd == 128) e = launch_rows<KVQ_Q8, 128>(plan, a, s);
    else if (hd == 256) e = launch_rows<KVQ_Q8, 256>(plan, a, s);
  } else if (fmt == KVQ_K8V4) {
    if (hd == 64) e = launch_rows<KVQ_K8V4, 64>(plan, a, s);
    else if (hd == 128) e = launch_rows<KVQ_K8V4, 128>(plan, a, s);
    else if (hd == 256) e = launch_rows<KVQ_K8V4, 256>(plan, a, s);
  }
  if (e != cudaSuccess) return e;
  if (hd == 64) return launch_combine<64>(a, s);
  if (hd == 128) return launch_combine<128>(a, s);
  return launch_combine<256>(a, s);
}

}  // namespace kvq

// kvq_chunk.cu -- attention of a prompt chunk over the contiguous fp16
// staging, on tensor cores.
//
// #3084 qwen35: FP16 K/V cache by default, int8 with --kv-q8, "Extra Notes":
// k_kv_f16 compacts a sequence into the [kvh][P][HD] fp16 halves that the
// prompt chunk's Q K^T and P V products read.  The chunk's T tokens are the
// sequence's last T cells (appended before the attention, as the decode
// step appends before it attends), so token t attends to cells
// [0, P - T + t]; query head h reads KV head h / (n_q / n_kv).
//
// Two kernels: head_dim 64 and 128 run on the fifth-generation tensor cores
// (chunk_attn_tc below); head_dim 256, whose q halves alone would fill an
// SM's shared memory there, runs on mma.sync (chunk_attn, described here).
//
// One CTA of 4 warps per (64 query rows, KV head); a row is a (chunk token,
// head of the GQA group) pair, so the G heads of a token share every K/V
// tile.  Each warp owns 16 rows and walks the key tiles its rows can see:
//
//   copies    64-key K and V tiles arrive by TMA (one tensor map per
//             128-byte span of a row, 128-byte swizzle) through a ring of 2
//             stages; an mbarrier per stage counts the bytes in, and the
//             warp that releases a stage last issues its refill.
//   q.k       S = Q K^T with mma.sync.m16n8k16 (f16 in, f32 accumulate); q
//             (times sm_scale * log2(e)) enters as fp16 hi + lo, about 22
//             significant bits, K as the exact staging values.
//   softmax   online, in the log2 domain, with a lazily raised reference
//             maximum; the causal mask is applied only on tiles that cross a
//             row's limit.
//   p.v       O += P V, P taken straight from the S accumulators (the C
//             fragment of two 8-key tiles is the A fragment of a 16-key
//             step) as fp16 hi + lo, V through ldmatrix.trans.
//
// Every mbarrier wait is bounded; a lost wait turns the CTA's rows into NaN
// and thread 0 still drains its own copies before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "kvq_internal.cuh"
#include "kvq_ptx.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr int kWarps = 4;
constexpr int kThr = kWarps * 32;
constexpr int kBM = 16 * kWarps;  // query rows per CTA
constexpr int kBN = 64;           // keys per stage
constexpr int kStages = 2;
constexpr float kTauC = 8.0f;     // lazy rescale threshold (log2 units)
constexpr unsigned kAll = 0xffffffffu;

template <int HD>
struct ChunkCfg {
  static constexpr int ROWB = HD * 2;         // staging bytes per row
  static constexpr int NSP = ROWB / 128;      // 128-byte swizzle spans per row
  static constexpr int TILE_B = kBN * ROWB;   // one K (or V) tile
  static constexpr int STAGE_B = 2 * TILE_B;  // K then V
  static constexpr int QROW = HD * 2 + 16;    // padded q row in shared memory
  static constexpr int SMEM_Q = kStages * STAGE_B;
  static constexpr int Q_B = 2 * kBM * QROW;  // hi rows, then lo rows
  static constexpr int SMEM_BAR = SMEM_Q + Q_B;
  static constexpr int SMEM_REL = SMEM_BAR + kStages * 8;
  static constexpr int SMEM = SMEM_REL + 16 + 1024;  // + 1 KB alignment slack
};

struct ChunkMaps {
  CUtensorMap k[4];
  CUtensorMap v[4];
};

// Swizzled offset of byte `b` of key row `c` (0..63) in a tile laid out
// [span][64 rows][128 bytes] (128-byte swizzle: 16-byte chunk ^= row & 7).
__device__ __forceinline__ uint32_t swz(int c, int b) {
  return (uint32_t)((b >> 7) * (kBN * 128) + c * 128) + ((uint32_t)(((b >> 4) & 7) ^ (c & 7)) << 4) +
         (uint32_t)(b & 15);
}

// CTAs per SM the shared memory allows (HD 64: 4, 128: 2, 256: 1), which
// sets the register budget
template <int HD>
__global__ void __launch_bounds__(kThr, HD == 64 ? 4 : (HD == 128 ? 2 : 1))
    chunk_attn(const __grid_constant__ ChunkMaps maps, ChunkArgs a) {
  using C = ChunkCfg<HD>;
  constexpr int KS = HD / 16;  // k-steps of q.k, n-tile pairs of p.v
  constexpr float kNegInf = -INFINITY;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::SMEM_BAR;
  int* s_rel = reinterpret_cast<int*>(smem + C::SMEM_REL);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kvh = blockIdx.y;
  const int r0 = blockIdx.x * kBM;         // first row of the CTA
  const int n_rows = a.T * a.G;
  const int P0 = a.P - a.T;                // cells before the chunk
  // keys the CTA's last row sees: [0, P0 + t_last]
  const int t_last = min(a.T - 1, (min(r0 + kBM, n_rows) - 1) / a.G);
  const int n_tiles = (P0 + t_last + 1 + kBN - 1) / kBN;
  const bool producer = threadIdx.x == 0;

  auto issue = [&](int it) {
    const int s = it % kStages;
    const uint32_t full = bar_full + 8 * s;
    mbar_expect_tx(full, (uint32_t)C::STAGE_B);
    const uint32_t st = sbase + s * C::STAGE_B;
    const int row = kvh * a.P + it * kBN;
#pragma unroll
    for (int sp = 0; sp < C::NSP; ++sp) {
      tma_load_2d(st + sp * kBN * 128, &maps.k[sp], 0, row, full);
      tma_load_2d(st + C::TILE_B + sp * kBN * 128, &maps.v[sp], 0, row, full);
    }
  };

  // thread 0 starts the first stages; meanwhile all threads bring the
  // CTA's q rows to shared memory as fp16 hi + lo, 16 values at a time
  if (producer) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.k[0])) : "memory");
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      s_rel[s] = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int it = 0; it < kStages && it < n_tiles; ++it) issue(it);
  }
  {
    constexpr int QPT = kBM * HD / kThr;  // q values per thread
    constexpr int QB = 16;                // per batch
    unsigned char* qs = smem + C::SMEM_Q;
#pragma unroll 1
    for (int u0 = 0; u0 < QPT; u0 += QB) {
      float qv[QB];
#pragma unroll
      for (int u = 0; u < QB; ++u) {
        const int i = threadIdx.x + (u0 + u) * kThr;
        const int r = i / HD, d = i - r * HD;
        const int gr = r0 + r;
        qv[u] = 0.f;
        if (gr < n_rows) {
          const int tok = gr / a.G, gg = gr - tok * a.G;
          qv[u] = __ldg(a.q + ((size_t)tok * a.n_q + (size_t)kvh * a.G + gg) * HD + d);
        }
      }
#pragma unroll
      for (int u = 0; u < QB; ++u) {
        const int i = threadIdx.x + (u0 + u) * kThr;
        const int r = i / HD, d = i - r * HD;
        const float x = qv[u] * a.qscale;
        const __half h = __float2half_rn(x);
        const __half lo = __float2half_rn(x - __half2float(h));
        *reinterpret_cast<__half*>(qs + r * C::QROW + d * 2) = h;
        *reinterpret_cast<__half*>(qs + (kBM + r) * C::QROW + d * 2) = lo;
      }
    }
  }
  __syncthreads();

  // ldmatrix lane addresses.  q (A of q.k): matrices (rows +0, dims lo),
  // (rows +8, dims lo), (rows +0, dims hi), (rows +8, dims hi).
  const int mi = lane >> 3, rr = lane & 7;
  const uint32_t q_lane = sbase + C::SMEM_Q + (uint32_t)(warp * 16 + (mi & 1) * 8 + rr) * C::QROW +
                          (uint32_t)(mi >> 1) * 16;
  // K (B of q.k, two 8-key n-tiles): matrices (keys +0, dims lo), (keys +0,
  // dims hi), (keys +8, dims lo), (keys +8, dims hi).
  const int kkey = (mi >> 1) * 8 + rr;
  const int kdb = (mi & 1) * 16;
  // V (B of p.v through .trans, two 8-dim n-tiles): matrices (keys +0, dims
  // lo), (keys +8, dims lo), (keys +0, dims hi), (keys +8, dims hi).
  const int vkey = (mi & 1) * 8 + rr;
  const int vdb = (mi >> 1) * 16;

  // causal limits of this thread's two rows (g and g + 8 of the warp)
  int lim[2];
  int lim_min = INT_MAX;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int gr = r0 + warp * 16 + g + 8 * j;
    lim[j] = gr < n_rows ? P0 + gr / a.G : -1;
  }
  {
    const int gr_first = r0 + warp * 16;  // the warp's smallest limit
    lim_min = gr_first < n_rows ? P0 + gr_first / a.G : -1;
  }
  // the warp's rows see no key past this tile
  const int gr_last = min(r0 + warp * 16 + 15, n_rows - 1);
  const int warp_tiles = gr_last >= r0 + warp * 16 ? (P0 + gr_last / a.G + 1 + kBN - 1) / kBN : 0;

  float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
  float o[HD / 8][4];
#pragma unroll
  for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  bool lost = false;
  for (int it = 0; it < n_tiles; ++it) {
    const int s = it % kStages;
    if (!mbar_wait(bar_full + 8 * s, (it / kStages) & 1)) lost = true;
    lost = __any_sync(kAll, lost);
    const uint32_t kt = sbase + s * C::STAGE_B;
    const uint32_t vt = kt + C::TILE_B;
    const int key0 = it * kBN;
    if (!lost && it < warp_tiles) {
      // ---------------- S = Q K^T (16 rows x 64 keys) ----------------
      float sacc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t qh[4], ql[4];
        ldsm_x4(qh, q_lane + ks * 32);
        ldsm_x4(ql, q_lane + kBM * C::QROW + ks * 32);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          uint32_t kb[4];
          ldsm_x4(kb, kt + swz(jj * 16 + kkey, ks * 32 + kdb));
          mma16816(sacc[2 * jj], qh, kb[0], kb[1]);
          mma16816(sacc[2 * jj], ql, kb[0], kb[1]);
          mma16816(sacc[2 * jj + 1], qh, kb[2], kb[3]);
          mma16816(sacc[2 * jj + 1], ql, kb[2], kb[3]);
        }
      }
      // ---------------- mask, online softmax ----------------
      const bool need_mask = key0 + kBN - 1 > lim_min;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (need_mask) {
#pragma unroll
          for (int n = 0; n < 8; ++n) {
            const int kabs = key0 + n * 8 + 2 * t;
            if (kabs > lim[j]) sacc[n][2 * j] = kNegInf;
            if (kabs + 1 > lim[j]) sacc[n][2 * j + 1] = kNegInf;
          }
        }
        float tmax = kNegInf;
#pragma unroll
        for (int n = 0; n < 8; ++n) tmax = fmaxf(tmax, fmaxf(sacc[n][2 * j], sacc[n][2 * j + 1]));
        tmax = fmaxf(tmax, __shfl_xor_sync(kAll, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(kAll, tmax, 2));
        if (tmax > m[j] + kTauC) {  // also true for the first finite maximum
          const float alpha = m[j] == kNegInf ? 0.f : fast_exp2(m[j] - tmax);
          m[j] = tmax;
          l[j] *= alpha;
#pragma unroll
          for (int n = 0; n < HD / 8; ++n) {
            o[n][2 * j] *= alpha;
            o[n][2 * j + 1] *= alpha;
          }
        }
        const bool none = m[j] == kNegInf;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const float p0 = none ? 0.f : fast_exp2(sacc[n][2 * j] - m[j]);
          const float p1 = none ? 0.f : fast_exp2(sacc[n][2 * j + 1] - m[j]);
          sacc[n][2 * j] = p0;
          sacc[n][2 * j + 1] = p1;
          l[j] += p0 + p1;
        }
      }
      // ---------------- O += P V ----------------
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t ph[4], pl[4];
        split_pair(sacc[2 * kk][0], sacc[2 * kk][1], ph[0], pl[0]);
        split_pair(sacc[2 * kk][2], sacc[2 * kk][3], ph[1], pl[1]);
        split_pair(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1], ph[2], pl[2]);
        split_pair(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
        for (int dn = 0; dn < KS; ++dn) {
          uint32_t vb[4];
          ldsm_x4_t(vb, vt + swz(kk * 16 + vkey, dn * 32 + vdb));
          mma16816(o[2 * dn], ph, vb[0], vb[1]);
          mma16816(o[2 * dn], pl, vb[0], vb[1]);
          mma16816(o[2 * dn + 1], ph, vb[2], vb[3]);
          mma16816(o[2 * dn + 1], pl, vb[2], vb[3]);
        }
      }
    }
    // release the stage; the last warp out refills it
    __syncwarp();
    if (lane == 0) {
      int prev;
      asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                   : "=r"(prev)
                   : "r"(smem_u32(s_rel + s))
                   : "memory");
      if (prev == kWarps - 1) {
        s_rel[s] = 0;
        if (it + kStages < n_tiles) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          issue(it + kStages);
        }
      }
    }
    if (lost) break;
  }
  if (producer) {
    // every copy this CTA issued has landed before it exits
    for (int it = n_tiles > kStages ? n_tiles - kStages : 0; it < n_tiles; ++it)
      (void)mbar_wait(bar_full + 8 * (it % kStages), (it / kStages) & 1);
  }

  // ---------------- normalise and write the rows ----------------
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    l[j] += __shfl_xor_sync(kAll, l[j], 1);
    l[j] += __shfl_xor_sync(kAll, l[j], 2);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int gr = r0 + warp * 16 + g + 8 * j;
    if (gr >= n_rows) continue;
    const int tok = gr / a.G, gg = gr - tok * a.G;
    float* orow = a.out + ((size_t)tok * a.n_q + (size_t)kvh * a.G + gg) * HD;
    const float inv = l[j] > 0.f ? 1.f / l[j] : 0.f;
    const float nan = __int_as_float(0x7fc00000);
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) {
      const float x0 = lost ? nan : o[n][2 * j] * inv;
      const float x1 = lost ? nan : o[n][2 * j + 1] * inv;
      *reinterpret_cast<float2*>(orow + n * 8 + 2 * t) = make_float2(x0, x1);
    }
  }
}


// ---------------------------------------------------------------------------
// head_dim 64 and 128 on the fifth-generation tensor cores (tcgen05, TMEM).
//
// One CTA per (128 query rows, KV head), six warps:
//   warps 0-3  softmax: thread i owns query row i = TMEM lane i.  It loads
//              its row of S from tensor memory, masks, keeps the running
//              maximum (raised lazily; the rare raise rescales its row of O
//              in tensor memory after the previous P V has finished), writes
//              P = 2^(S - m) as fp16 over the first 64 columns of the same
//              S buffer, and at the end divides its row of O by the sum.
//   warp 4     TMA producer: 128-key K and V tiles (two stages each; a
//              tile is head_dim / 64 boxes of 128 bytes by 128 rows).
//   warp 5     allocates the 512 TMEM columns and issues the MMAs from one
//              thread: S_j = Q K_j^T (M = N = 128, fp32 in TMEM, three S
//              buffers) as Q_hi K^T + Q_lo K^T, and O += P_j V_j with P read
//              from tensor memory and V as an MN-major operand.
// The issue order S_0, S_1, PV_0, S_2, PV_1, S_3, ... keeps the tensor pipe
// fed while the softmax of one tile overlaps the MMAs of its neighbours.
// q * sm_scale * log2(e) enters as fp16 hi + lo (the logits need the bits:
// K's large channels magnify q's rounding), p as one fp16 value.
// ---------------------------------------------------------------------------
namespace tcc {
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kSoftWarps = 4;
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;
constexpr int SPAN_B = BN * 128;            // one 128-byte span of a 128-row tile
// barriers
constexpr int KFULL = 0, KEMPTY = 2, VFULL = 4, VEMPTY = 6, SFULL = 8, PFULL = 11, SFREE = 14,
              ODONE = 17, QREADY = 18, NBAR = 19;
constexpr uint32_t TMEM_COLS = 512;             // S buffers at columns 0, 128, 256; O at 384
constexpr uint32_t COL_O = 384;

// Shared memory of the head_dim-HD kernel: q hi and lo, two K and two V
// stages, each a tile of HD / 64 spans ([span][row][128 B], 128-byte
// swizzle), then the barriers and the tensor-memory address slot.
template <int HD>
struct TcLayout {
  static constexpr int NSP = HD / 64;               // 128-byte spans per row
  static constexpr int TILE_B = NSP * SPAN_B;       // 128 rows x 2 HD bytes
  static constexpr int OFF_QH = 0, OFF_QL = TILE_B;
  static constexpr int OFF_K = 2 * TILE_B;          // two K stages
  static constexpr int OFF_V = OFF_K + 2 * TILE_B;  // two V stages
  static constexpr int OFF_BAR = OFF_V + 2 * TILE_B;
  static constexpr int OFF_TSLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TSLOT + 16 + 1024;   // + alignment slack
  static_assert(HD == 64 || HD == 128, "q hi + lo and two K and V stages fit one SM up to head_dim 128");
  static_assert(SMEM <= 227 * 1024, "one CTA per SM");
  static_assert(COL_O + HD <= TMEM_COLS, "O fits tensor memory beside the three S buffers");
};

// byte offset of (row r, byte b) of a [span][128 rows][128 B] tile
__device__ __forceinline__ uint32_t sw(int r, int b) {
  return (uint32_t)((b >> 7) * SPAN_B + r * 128) + ((uint32_t)(((b >> 4) & 7) ^ (r & 7)) << 4) +
         (uint32_t)(b & 15);
}
}  // namespace tcc

template <int HD>
__global__ void __launch_bounds__(tcc::kThreads, 1)
    chunk_attn_tc(const __grid_constant__ ChunkMaps maps, ChunkArgs a) {
  using namespace tcc;
  using Lay = TcLayout<HD>;
  constexpr int TILE_B = Lay::TILE_B, OFF_QH = Lay::OFF_QH, OFF_QL = Lay::OFF_QL, OFF_K = Lay::OFF_K,
                OFF_V = Lay::OFF_V, OFF_BAR = Lay::OFF_BAR, OFF_TSLOT = Lay::OFF_TSLOT;
  constexpr float kNegInf = -INFINITY;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8 * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y;
  const int r0 = blockIdx.x * BM;
  const int n_rows = a.T * a.G;
  const int P0 = a.P - a.T;                 // cells before the chunk
  const int t_last = min(a.T - 1, (min(r0 + BM, n_rows) - 1) / a.G);
  const int n_tiles = (P0 + t_last + 1 + BN - 1) / BN;   // key tiles the CTA's rows see

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(KFULL + i), 1);
      mbar_init(bar(KEMPTY + i), 1);
      mbar_init(bar(VFULL + i), 1);
      mbar_init(bar(VEMPTY + i), 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(bar(SFULL + i), 1);
      mbar_init(bar(PFULL + i), kSoftWarps * 32);
      mbar_init(bar(SFREE + i), 1);
    }
    mbar_init(bar(ODONE), 1);
    mbar_init(bar(QREADY), kSoftWarps * 32);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(sbase + OFF_TSLOT, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TSLOT);
  bool lost = false;

  if (warp == kProdWarp) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.k[0])) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.v[0])) : "memory");
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j & 1;
        const int row = kvh * a.P + j * BN;
        if (j >= 2 && !mbar_wait(bar(KEMPTY + s), ((j >> 1) - 1) & 1)) break;
        mbar_expect_tx(bar(KFULL + s), (uint32_t)TILE_B);
#pragma unroll
        for (int sp = 0; sp < Lay::NSP; ++sp)
          tma_load_2d(sbase + OFF_K + s * TILE_B + sp * SPAN_B, &maps.k[sp], 0, row, bar(KFULL + s));
        if (j >= 2 && !mbar_wait(bar(VEMPTY + s), ((j >> 1) - 1) & 1)) break;
        mbar_expect_tx(bar(VFULL + s), (uint32_t)TILE_B);
#pragma unroll
        for (int sp = 0; sp < Lay::NSP; ++sp)
          tma_load_2d(sbase + OFF_V + s * TILE_B + sp * SPAN_B, &maps.v[sp], 0, row, bar(VFULL + s));
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t IS = umma_idesc_f16(BM, BN, false, false);   // Q, K both K-major
      constexpr uint32_t IO = umma_idesc_f16(BM, HD, false, true);   // P (TMEM), V MN-major
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1, b = j % 3;
        if (!mbar_wait(bar(KFULL + s), (j >> 1) & 1)) return false;
        if (j >= 3 && !mbar_wait(bar(SFREE + b), (j / 3 - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)b * 128;
#pragma unroll
        for (int hl = 0; hl < 2; ++hl)
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (uint32_t)(kk >> 2) * SPAN_B + (uint32_t)(kk & 3) * 32;
            umma_ss(d, umma_desc_sw128(sbase + (hl ? OFF_QL : OFF_QH) + off, 16, 1024),
                    umma_desc_sw128(sbase + OFF_K + s * TILE_B + off, 16, 1024), IS, hl + kk > 0);
          }
        umma_commit(bar(SFULL + b));
        umma_commit(bar(KEMPTY + s));
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int s = j & 1, b = j % 3;
        if (!mbar_wait(bar(PFULL + b), (j / 3) & 1)) return false;
        if (!mbar_wait(bar(VFULL + s), (j >> 1) & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)   // 16 keys: P columns 8 kk .. + 7, two V atoms
          umma_ts(tmem + COL_O, tmem + (uint32_t)b * 128 + (uint32_t)kk * 8,
                  umma_desc_sw128(sbase + OFF_V + s * TILE_B + kk * 2048, SPAN_B, 1024), IO,
                  j > 0 || kk > 0);
        umma_commit(bar(SFREE + b));
        umma_commit(bar(VEMPTY + s));
        umma_commit(bar(ODONE));
        return true;
      };
      bool ok = mbar_wait(bar(QREADY), 0);
      if (ok) {
        tc_fence_after();
        ok = issue_s(0) && (n_tiles < 2 || issue_s(1));
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        ok = issue_pv(j);
        if (ok && j + 2 < n_tiles) ok = issue_s(j + 2);
      }
    }
  } else {
    // ---------------- softmax warps: thread = query row ----------------
    const int row = threadIdx.x;
    const int gr = r0 + row;
    const bool valid = gr < n_rows;
    const int tok = valid ? gr / a.G : 0;
    const int gg = valid ? gr - tok * a.G : 0;
    const int lim = valid ? P0 + tok : -1;                  // last key this row sees
    {
      // q * sm_scale * log2(e) -> fp16 hi + lo rows of the A operand
      const float* qrow = a.q + ((size_t)tok * a.n_q + (size_t)kvh * a.G + gg) * HD;
#pragma unroll 4
      for (int c = 0; c < HD / 8; ++c) {
        float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
        if (valid) {
          x0 = __ldg(reinterpret_cast<const float4*>(qrow + 8 * c));
          x1 = __ldg(reinterpret_cast<const float4*>(qrow + 8 * c + 4));
        }
        const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          split_pair(x[2 * e] * a.qscale, x[2 * e + 1] * a.qscale, hi[e], lo[e]);
        *reinterpret_cast<uint4*>(smem + OFF_QH + sw(row, c * 16)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(smem + OFF_QL + sw(row, c * 16)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(QREADY)) : "memory");
    }
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float m = -1e30f, l = 0.f;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j % 3;
      lost = __any_sync(kAll, !mbar_wait(bar(SFULL + b), (j / 3) & 1));
      if (lost) break;
      tc_fence_after();
      float sv[BN];
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32)
        tmem_ld32(tmem + lane_base + (uint32_t)b * 128 + c0, *reinterpret_cast<uint32_t(*)[32]>(sv + c0));
      tmem_wait_ld();
      const int key0 = j * BN;
      if (key0 + BN - 1 > lim) {   // keys past this row's causal limit
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (key0 + c > lim) sv[c] = kNegInf;
      }
      // the row maximum and (below) the row sum over 8 independent
      // chains: a single chain of 127 dependent steps is what one warp per
      // scheduler cannot hide
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = sv[e];
#pragma unroll
      for (int c = 8; c < BN; c += 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(mx8[e], sv[c + e]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const bool rise = mx > m + kTauC;
      float alpha = 1.f;
      if (rise) {
        alpha = fast_exp2(m - mx);   // 0 from the finite start
        m = mx;
        l *= alpha;
      }
      if (j > 0 && __any_sync(kAll, rise)) {
        // O holds P V of the tiles so far: wait for the last one, rescale
        lost = __any_sync(kAll, !mbar_wait(bar(ODONE), (j - 1) & 1));
        if (lost) break;
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < HD; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + COL_O + c0, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(tmem + lane_base + COL_O + c0, ov);
        }
      }
      float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int h = 0; h < 2; ++h) {   // keys 64 h .. + 63 -> P columns 32 h .. + 31
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = fast_exp2(sv[64 * h + 2 * e] - m);
          const float p1 = fast_exp2(sv[64 * h + 2 * e + 1] - m);
          sum8[e & 7] += p0 + p1;
          pk[e] = pack_half2(p0, p1);
        }
        tmem_st32(tmem + lane_base + (uint32_t)b * 128 + 32 * h, pk);
      }
      l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      tmem_wait_st();
      tc_fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(PFULL + b)) : "memory");
    }
    if (!lost && n_tiles > 0) lost = __any_sync(kAll, !mbar_wait(bar(ODONE), (n_tiles - 1) & 1));
    tc_fence_after();
    float* orow = a.out + ((size_t)tok * a.n_q + (size_t)kvh * a.G + gg) * HD;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c0 = 0; c0 < HD; c0 += 32) {
      uint32_t ov[32];
      tmem_ld32(tmem + lane_base + COL_O + c0, ov);
      tmem_wait_ld();
      if (valid) {
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float4 r4 = make_float4(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv,
                                  __uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
          if (lost) {
            const float nan = __int_as_float(0x7fc00000);
            r4 = make_float4(nan, nan, nan, nan);
          }
          *reinterpret_cast<float4*>(orow + c0 + e) = r4;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// One 2D tensor map per 128-byte span of a staging row: [n_kv * P rows]
// [128 bytes], row stride HD * 2 bytes, box 128 bytes x box_rows rows.
bool make_span_map(CUtensorMap* map, const void* base, int sp, long long rows, int row_bytes,
                   int box_rows = kBN) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  void* span = static_cast<char*>(const_cast<void*>(base)) + (size_t)sp * 128;
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, span, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD>
cudaError_t launch_hd(const ChunkArgs& a, cudaStream_t s) {
  using C = ChunkCfg<HD>;
  // the dynamic shared-memory limit, raised once per context
  static ContextCache<int> limit_set;
  int done = 0;
  if (!per_context(limit_set, &done, [](int* v) {
        *v = 1;
        return cudaFuncSetAttribute(chunk_attn<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::SMEM) == cudaSuccess;
      }))
    return cudaErrorInvalidConfiguration;
  ChunkMaps maps;
  memset(&maps, 0, sizeof(maps));
  const long long rows = (long long)a.n_kv * a.P;
  for (int sp = 0; sp < C::NSP; ++sp) {
    if (!make_span_map(&maps.k[sp], a.k16, sp, rows, C::ROWB) ||
        !make_span_map(&maps.v[sp], a.v16, sp, rows, C::ROWB))
      return cudaErrorInvalidValue;
  }
  const long long row_tiles = ((long long)a.T * a.G + kBM - 1) / kBM;
  if (row_tiles > 0x7fffffffLL || a.n_kv > 65535) return cudaErrorInvalidValue;
  chunk_attn<HD><<<dim3((unsigned)row_tiles, (unsigned)a.n_kv), kThr, C::SMEM, s>>>(maps, a);
  return cudaGetLastError();
}


// head_dim 64 and 128: the tcgen05 kernel, one CTA of 192 threads per (128
// rows, KV head), 128-key tiles.
template <int HD>
cudaError_t launch_tc(const ChunkArgs& a, cudaStream_t s) {
  using Lay = tcc::TcLayout<HD>;
  static ContextCache<int> limit_set;
  int done = 0;
  if (!per_context(limit_set, &done, [](int* v) {
        *v = 1;
        return cudaFuncSetAttribute(chunk_attn_tc<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Lay::SMEM) == cudaSuccess;
      }))
    return cudaErrorInvalidConfiguration;
  ChunkMaps maps;
  memset(&maps, 0, sizeof(maps));
  const long long rows = (long long)a.n_kv * a.P;
  for (int sp = 0; sp < Lay::NSP; ++sp) {
    if (!make_span_map(&maps.k[sp], a.k16, sp, rows, HD * 2, tcc::BN) ||
        !make_span_map(&maps.v[sp], a.v16, sp, rows, HD * 2, tcc::BN))
      return cudaErrorInvalidValue;
  }
  const long long row_tiles = ((long long)a.T * a.G + tcc::BM - 1) / tcc::BM;
  if (row_tiles > 0x7fffffffLL || a.n_kv > 65535) return cudaErrorInvalidValue;
  chunk_attn_tc<HD><<<dim3((unsigned)row_tiles, (unsigned)a.n_kv), tcc::kThreads, Lay::SMEM, s>>>(maps, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_attn(int hd, const ChunkArgs& a, cudaStream_t s) {
  switch (hd) {
    case 64: return launch_tc<64>(a, s);
    case 128: return launch_tc<128>(a, s);
    case 256: return launch_hd<256>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq

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
// One kernel, on the fifth-generation tensor cores (tcgen05: operands
// staged by TMA in shared memory, fp32 accumulators in tensor memory); it
// is described above chunk_attn_tc below.  Every mbarrier wait is bounded:
// a lost wait turns the CTA's rows into NaN, and the copies in flight land
// before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include "kvq_internal.cuh"
#include "kvq_key_splits.h"
#include "kvq_ptx.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr float kTauC = 8.0f;     // lazy rescale threshold (log2 units)
constexpr unsigned kAll = 0xffffffffu;

struct ChunkMaps {
  CUtensorMap k[4];
  CUtensorMap v[4];
};

// ---------------------------------------------------------------------------
// The chunk attention on the fifth-generation tensor cores (tcgen05, TMEM).
//
// One CTA per (128 query rows, KV head); a row is a (chunk token, head of
// the GQA group) pair, so the G heads of a token share every K/V tile.  The
// key tiles are BN = 128 keys at head_dim 64 and 128, 64 at 256.
//   warps 0-3  softmax: thread i owns query row i = TMEM lane i.  It loads
//              its row of S from tensor memory, masks (only on tiles that
//              cross a row's causal limit), keeps the running maximum in
//              the log2 domain (raised lazily; the rare raise rescales its
//              row of O in tensor memory after the previous P V has
//              finished), writes P = 2^(S - m) as fp16 over the first BN / 2
//              columns of the same S buffer, and at the end divides its row
//              of O by the sum.
//   warp 4     TMA producer of the K tiles (two stages; a tile is
//              head_dim / 64 boxes of 128 bytes by BN rows, 128-byte
//              swizzle), and of the V tiles too at head_dim 64 and 128 (two
//              stages); at 256, V has one stage and warp 7 fetches it.
//   warp 5     allocates the 512 TMEM columns; one thread issues
//              S_j = Q K_j^T (M = 128, N = BN, fp32 in TMEM, three S
//              buffers) as Q_hi K^T + Q_lo K^T, up to three tiles ahead.
//   warp 6     one thread issues O += P_j V_j (N = head_dim) with P read
//              from tensor memory and V as an MN-major operand.
// Two issuing threads keep the tensor pipe fed: it holds only an MMA or two
// beyond the last one issued, so while one thread checks its barriers the
// other's MMAs run, and the softmax of one tile overlaps the MMAs of its
// neighbours.
// q * sm_scale * log2(e) enters as fp16 hi + lo (about 22 significant bits:
// K's large channels magnify q's rounding), K and V as the exact staging
// values, p as one fp16 value.
// ---------------------------------------------------------------------------
namespace tcc {
constexpr int BM = 128;
constexpr int kSoftWarps = 4;
constexpr int kProdWarp = 4;    // K tiles (and V tiles unless a warp of their own)
constexpr int kMmaWarp = 5;     // S MMAs; owns the tensor memory
constexpr int kPvWarp = 6;      // P V MMAs
constexpr int kProdWarpV = 7;   // V tiles, when V has a single stage
constexpr int QSPAN_B = BM * 128;   // one 128-byte span of the 128 q rows
// barriers.  SFREE[b] completes when the P V product that read S buffer b
// has (so the rescale of O before tile j's P waits on SFREE[(j - 1) % 3]:
// never more than one phase behind, as the S MMAs of tile j - 1 waited for
// the product three tiles before it).  ALLDONE completes once, after the
// last product: when the last p is written, the last two products can still
// be running, one more than a parity wait on a per-tile barrier tells apart.
// SDRAIN / PDRAIN: each issuing thread's last commit, waited on before the
// tensor memory is freed (after a lost wait too).
constexpr int KFULL = 0, KEMPTY = 2, VFULL = 4, VEMPTY = 6, SFULL = 8, PFULL = 11, SFREE = 14,
              QREADY = 17, ALLDONE = 18, SDRAIN = 19, PDRAIN = 20, NBAR = 21;
constexpr uint32_t TMEM_COLS = 512;

// The head_dim-HD kernel's tiles and memory.  Shared memory: q hi and lo
// (HD / 64 spans of 128 rows, [span][row][128 B], 128-byte swizzle), KST K
// and VST V stages of BN keys, the barriers, the tensor-memory address
// slot.  Tensor memory: three S buffers of BN columns, then O (HD columns).
// Head dims 64 and 128 take 128-key tiles and two stages of each; at 256
// the q halves take 128 KB, so the key tiles are 64 keys, K has two stages
// and V one, fetched by a warp of its own.
template <int HD>
struct TcLayout {
  static constexpr int BN = HD == 256 ? 64 : 128;     // keys per tile
  static constexpr int KST = 2, VST = HD == 256 ? 1 : 2;
  static constexpr bool SPLIT_PROD = VST == 1;        // V from warp 7
  static constexpr int THREADS = SPLIT_PROD ? 256 : 224;
  static constexpr int NSP = HD / 64;                 // 128-byte spans per row
  static constexpr int QTILE_B = NSP * QSPAN_B;       // 128 q rows x 2 HD bytes
  static constexpr int KSPAN_B = BN * 128;            // one span of a key tile
  static constexpr int KTILE_B = NSP * KSPAN_B;       // BN key rows x 2 HD bytes
  static constexpr int OFF_QH = 0, OFF_QL = QTILE_B;
  static constexpr int OFF_K = 2 * QTILE_B;
  static constexpr int OFF_V = OFF_K + KST * KTILE_B;
  static constexpr int OFF_BAR = OFF_V + VST * KTILE_B;
  static constexpr int OFF_TSLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TSLOT + 16 + 1024;   // + alignment slack
  static constexpr uint32_t COL_O = 3 * BN;           // after the three S buffers
  static_assert(HD == 64 || HD == 128 || HD == 256, "head dims");
  static_assert(SMEM <= 227 * 1024, "one CTA per SM");
  static_assert(COL_O + HD <= TMEM_COLS, "O fits tensor memory beside the three S buffers");
  static_assert(KSPAN_B % 1024 == 0 && QTILE_B % 1024 == 0, "swizzle atoms stay 1 KB aligned");
};

// byte offset of (row r, byte b) of a [span][128 rows][128 B] q tile
__device__ __forceinline__ uint32_t sw(int r, int b) {
  return (uint32_t)((b >> 7) * QSPAN_B + r * 128) + ((uint32_t)(((b >> 4) & 7) ^ (r & 7)) << 4) +
         (uint32_t)(b & 15);
}
}  // namespace tcc

// LW: the lost-wait test's instantiation, whose waits take their poll limit
// from the call and whose stages expect a.extra_tx bytes more than any copy
// delivers; the ordinary one keeps the constant limit in its hot loops.
template <int HD, bool LW>
__global__ void __launch_bounds__(tcc::TcLayout<HD>::THREADS, 1)
    chunk_attn_tc(const __grid_constant__ ChunkMaps maps, ChunkArgs a) {
  using namespace tcc;
  using Lay = TcLayout<HD>;
  constexpr int BN = Lay::BN, KST = Lay::KST, VST = Lay::VST;
  constexpr int KTILE_B = Lay::KTILE_B, KSPAN_B = Lay::KSPAN_B, OFF_QH = Lay::OFF_QH,
                OFF_QL = Lay::OFF_QL, OFF_K = Lay::OFF_K, OFF_V = Lay::OFF_V, OFF_BAR = Lay::OFF_BAR,
                OFF_TSLOT = Lay::OFF_TSLOT;
  constexpr uint32_t COL_O = Lay::COL_O;
  constexpr float kNegInf = -INFINITY;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8 * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y;
  const uint32_t wl = LW ? a.wait_limit : kDefaultWaitLimit;   // polls before a wait is lost
  const uint32_t extra_tx = LW ? a.extra_tx : 0u;
  // row tiles in descending order: the last ones (later tokens) see the
  // most keys, so the longest CTAs start first and the grid's last, partial
  // wave holds the shortest
  const int r0 = (int)(gridDim.x - 1 - blockIdx.x) * BM;
  const int n_rows = a.T * a.G;
  const int P0 = a.P - a.T;                 // cells before the chunk
  const int t_last = min(a.T - 1, (min(r0 + BM, n_rows) - 1) / a.G);
  const int n_all = (P0 + t_last + 1 + BN - 1) / BN;     // key tiles the CTA's rows see
  // key splits: the gridDim.z CTAs of a (row tile, KV head) form a cluster,
  // each takes a contiguous share of the key tiles, and they merge at the end
  const int n_split = (int)gridDim.z;
  const int per = (n_all + n_split - 1) / n_split;
  const int j0 = min(n_all, (int)blockIdx.z * per);     // this CTA's first key tile
  const int n_tiles = min(n_all, j0 + per) - j0;         // and its count (0 possible)

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
    mbar_init(bar(ALLDONE), 1);
    mbar_init(bar(SDRAIN), 1);
    mbar_init(bar(PDRAIN), 1);
    mbar_init(bar(QREADY), kSoftWarps * 32);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(sbase + OFF_TSLOT, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TSLOT);
  bool lost = false;
  // softmax threads: thread = query row (TMEM lane); the running maximum m
  // and sum l outlive the softmax section for the output and the merge
  const int row = threadIdx.x;
  const int gr = r0 + row;
  const bool valid = row < BM && gr < n_rows;
  const int tok = valid ? gr / a.G : 0;
  const int gg = valid ? gr - tok * a.G : 0;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  float m = -1e30f, l = 0.f;

  if (warp == kProdWarp || (Lay::SPLIT_PROD && warp == kProdWarpV)) {
    // K tiles from warp 4; V tiles from warp 4 too, or from warp 7 when V has
    // a single stage (its refill waits for P V, which must not hold K back)
    if (lane == 0) {
      const bool do_k = warp == kProdWarp, do_v = !Lay::SPLIT_PROD || warp == kProdWarpV;
      if (do_k) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.k[0])) : "memory");
      if (do_v) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.v[0])) : "memory");
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int ks = j % KST, vs = j % VST;
        const int krow = kvh * a.P + (j0 + j) * BN;   // first staging row of the tile
        if (do_k) {
          if (j >= KST && !mbar_wait(bar(KEMPTY + ks), (j / KST - 1) & 1, wl)) break;
          mbar_expect_tx(bar(KFULL + ks), (uint32_t)KTILE_B + extra_tx);
#pragma unroll
          for (int sp = 0; sp < Lay::NSP; ++sp)
            tma_load_2d(sbase + OFF_K + ks * KTILE_B + sp * KSPAN_B, &maps.k[sp], 0, krow, bar(KFULL + ks));
          k_issued = j + 1;
        }
        if (do_v) {
          if (j >= VST && !mbar_wait(bar(VEMPTY + vs), (j / VST - 1) & 1, wl)) break;
          mbar_expect_tx(bar(VFULL + vs), (uint32_t)KTILE_B + extra_tx);
#pragma unroll
          for (int sp = 0; sp < Lay::NSP; ++sp)
            tma_load_2d(sbase + OFF_V + vs * KTILE_B + sp * KSPAN_B, &maps.v[sp], 0, krow, bar(VFULL + vs));
          v_issued = j + 1;
        }
      }
      // every copy has landed before the CTA can exit (the waits return at
      // once in normal runs; they are bounded after a lost wait)
      for (int j = k_issued > KST ? k_issued - KST : 0; j < k_issued; ++j)
        (void)mbar_wait(bar(KFULL + j % KST), (j / KST) & 1, wl);
      for (int j = v_issued > VST ? v_issued - VST : 0; j < v_issued; ++j)
        (void)mbar_wait(bar(VFULL + j % VST), (j / VST) & 1, wl);
    }
  } else if (warp == kMmaWarp) {
    // S_j = Q_hi K_j^T + Q_lo K_j^T, up to three tiles ahead of the P V
    // products (one per S buffer)
    if (lane == 0) {
      constexpr uint32_t IS = umma_idesc_f16(BM, BN, false, false);   // Q, K both K-major
      // operand descriptors built once, stepped per MMA by constant offsets
      const uint64_t dq[2] = {umma_desc_sw128(sbase + OFF_QH, 16, 1024),
                              umma_desc_sw128(sbase + OFF_QL, 16, 1024)};
      const uint64_t dk0 = umma_desc_sw128(sbase + OFF_K, 16, 1024);
      bool ok = mbar_wait(bar(QREADY), 0, wl);
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int ks = j % KST, b = j % 3;
        ok = mbar_wait(bar(KFULL + ks), (j / KST) & 1, wl) &&
             (j < 3 || mbar_wait(bar(SFREE + b), (j / 3 - 1) & 1, wl));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * BN);
        const uint64_t dk = umma_desc_step(dk0, (uint32_t)(ks * KTILE_B));
#pragma unroll
        for (int hl = 0; hl < 2; ++hl)
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t in = (uint32_t)(kk & 3) * 32;   // 16 dims: 32 bytes into a span
            umma_ss(d, umma_desc_step(dq[hl], (kk >> 2) * QSPAN_B + in),
                    umma_desc_step(dk, (kk >> 2) * KSPAN_B + in), IS, hl + kk > 0);
          }
        umma_commit(bar(SFULL + b));
        umma_commit(bar(KEMPTY + ks));
      }
      // every MMA this thread issued has completed before the CTA frees the
      // tensor memory (at once in normal runs; bounded after a lost wait)
      umma_commit(bar(SDRAIN));
      (void)mbar_wait(bar(SDRAIN), 0, wl);
    }
  } else if (warp == kPvWarp) {
    // O += P_j V_j.  A thread of its own: while it waits for a tile's p,
    // the S thread keeps the tensor pipe fed, and the other way round (the
    // pipe holds only an MMA or two beyond the last one issued, so a single
    // issuing thread's barrier checks left it idle)
    if (lane == 0) {
      constexpr uint32_t IO = umma_idesc_f16(BM, HD, false, true);   // P (TMEM), V MN-major
      const uint64_t dv0 = umma_desc_sw128(sbase + OFF_V, KSPAN_B, 1024);
      bool ok = true;
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int vs = j % VST, b = j % 3;
        ok = mbar_wait(bar(PFULL + b), (j / 3) & 1, wl) && mbar_wait(bar(VFULL + vs), (j / VST) & 1, wl);
        if (!ok) break;
        tc_fence_after();
        const uint32_t pa = tmem + (uint32_t)(b * BN);
        const uint64_t dv = umma_desc_step(dv0, (uint32_t)(vs * KTILE_B));
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)   // 16 keys: P columns 8 kk .. + 7, two V atoms
          umma_ts(tmem + COL_O, pa + (uint32_t)kk * 8, umma_desc_step(dv, kk * 2048), IO, j > 0 || kk > 0);
        umma_commit(bar(SFREE + b));
        umma_commit(bar(VEMPTY + vs));
      }
      if (ok) umma_commit(bar(ALLDONE));   // every product above has completed
      umma_commit(bar(PDRAIN));
      (void)mbar_wait(bar(PDRAIN), 0, wl);
    }
  } else {
    // ---------------- softmax warps: thread = query row ----------------
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
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j % 3;
      lost = __any_sync(kAll, !mbar_wait(bar(SFULL + b), (j / 3) & 1, wl));
      if (lost) break;
      tc_fence_after();
      float sv[BN];
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32)
        tmem_ld32(tmem + lane_base + (uint32_t)(b * BN) + c0, *reinterpret_cast<uint32_t(*)[32]>(sv + c0));
      tmem_wait_ld();
      const int key0 = (j0 + j) * BN;
      if (key0 + BN - 1 > lim) {   // keys past this row's causal limit
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (key0 + c > lim) sv[c] = kNegInf;
      }
      // the row maximum and (below) the row sum over 8 independent
      // chains (a single chain of dependent steps is what one warp per
      // scheduler cannot hide); three-input maxima take two logits a step,
      // packed fp32 adds two subtractions or sums an instruction
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(sv[e], sv[8 + e]);
#pragma unroll
      for (int c = 16; c < BN; c += 16)
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = max3f(mx8[e], sv[c + e], sv[c + 8 + e]);
      const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7]));
      const bool rise = mx > m + kTauC;
      float alpha = 1.f;
      if (rise) {
        alpha = fast_exp2(m - mx);   // 0 from the finite start
        m = mx;
        l *= alpha;
      }
      if (j > 0 && __any_sync(kAll, rise)) {
        // O holds P V of the tiles so far: wait for the last one, rescale
        lost = __any_sync(kAll, !mbar_wait(bar(SFREE + (j - 1) % 3), ((j - 1) / 3) & 1, wl));
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
      const float nm = -m;
#pragma unroll
      for (int h = 0; h < BN / 64; ++h) {   // keys 64 h .. + 63 -> P columns 32 h .. + 31
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x0, x1;
          add_f32x2(x0, x1, sv[64 * h + 2 * e], sv[64 * h + 2 * e + 1], nm, nm);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          const int c = 2 * (e & 3);
          add_f32x2(sum8[c], sum8[c + 1], sum8[c], sum8[c + 1], p0, p1);
          pk[e] = pack_half2(p0, p1);
        }
        tmem_st32(tmem + lane_base + (uint32_t)(b * BN) + 32 * h, pk);
      }
      l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      tmem_wait_st();
      tc_fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(PFULL + b)) : "memory");
    }
    if (!lost && n_tiles > 0) lost = __any_sync(kAll, !mbar_wait(bar(ALLDONE), 0, wl));
  }
  // every copy and MMA of the CTA has completed (each role drained its own)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool soft = warp < kSoftWarps;
  float* orow = a.out + ((size_t)tok * a.n_q + (size_t)kvh * a.G + gg) * HD;
  const float nan = __int_as_float(0x7fc00000);
  if (n_split == 1) {
    if (soft) {
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
            if (lost) r4 = make_float4(nan, nan, nan, nan);
            *reinterpret_cast<float4*>(orow + c0 + e) = r4;
          }
        }
      }
    }
  } else {
    // Merge of the cluster's key splits through distributed shared memory
    // (the q and K stage areas are free now): (m, l) of every row first,
    // then each CTA's O scaled by 2^(m - M) / L, then each CTA sums a slice
    // of the columns over the cluster and writes it.  Every thread of every
    // CTA passes the three cluster barriers exactly once.
    float2* s_ml = reinterpret_cast<float2*>(smem + OFF_K);   // [BM]: (m, l) of each row
    const uint32_t s_o = sbase + OFF_QH;                     // [BM][HD] fp32, 16-byte chunks swizzled
    auto o_chunk = [&](int r, int ch) -> uint32_t {          // byte offset of chunk ch of row r
      return (uint32_t)(r * HD * 4) + ((uint32_t)(ch ^ (r & 7)) << 4);
    };
    if (soft) s_ml[row] = make_float2(m, lost ? nan : l);   // a lost wait: NaN through L
    cluster_sync_all();
    if (soft) {
      float M = -INFINITY;
      for (int z = 0; z < n_split; ++z) M = fmaxf(M, ld_dsmem_f32(smem_u32(&s_ml[row].x), z));
      float L = 0.f;
      for (int z = 0; z < n_split; ++z) {
        const float mz = ld_dsmem_f32(smem_u32(&s_ml[row].x), z), lz = ld_dsmem_f32(smem_u32(&s_ml[row].y), z);
        L += lz * fast_exp2(mz - M);
      }
      const float c = fast_exp2(m - M) / L;   // this split's weight (rows that see no key: unused)
#pragma unroll
      for (int c0 = 0; c0 < HD; c0 += 32) {
        uint32_t ov[32];
        if (n_tiles > 0) {
          tmem_ld32(tmem + lane_base + COL_O + c0, ov);
          tmem_wait_ld();
        }
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 r4 = n_tiles > 0
              ? make_float4(__uint_as_float(ov[e]) * c, __uint_as_float(ov[e + 1]) * c,
                            __uint_as_float(ov[e + 2]) * c, __uint_as_float(ov[e + 3]) * c)
              : make_float4(0.f, 0.f, 0.f, 0.f);
          st_shared_v4(s_o + o_chunk(row, (c0 + e) >> 2), r4);
        }
      }
    }
    cluster_sync_all();
    if (soft && valid) {
      // this CTA's slice of the row's 16-byte chunks, summed over the cluster
      constexpr int NCH = HD / 4;
      const int z0 = (int)blockIdx.z;
      const int ch_b = z0 * NCH / n_split, ch_e = (z0 + 1) * NCH / n_split;
      for (int ch = ch_b; ch < ch_e; ++ch) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int z = 0; z < n_split; ++z) {
          const float4 v4 = ld_dsmem_v4(s_o + o_chunk(row, ch), z);
          acc.x += v4.x;
          acc.y += v4.y;
          acc.z += v4.z;
          acc.w += v4.w;
        }
        *reinterpret_cast<float4*>(orow + 4 * ch) = acc;
      }
    }
    cluster_sync_all();   // no CTA leaves while a peer reads its shared memory
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
                   int box_rows) {
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

// The cluster launch of chunk_attn_tc<HD> with n_split CTAs per cluster
// (along z); 1: a plain launch.
template <int HD>
cudaLaunchConfig_t tc_config(dim3 grid, int n_split, cudaStream_t s, cudaLaunchAttribute* attr) {
  using Lay = tcc::TcLayout<HD>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Lay::THREADS);
  cfg.dynamicSmemBytes = Lay::SMEM;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)n_split;
  cfg.attrs = attr;
  cfg.numAttrs = n_split > 1 ? 1 : 0;
  return cfg;
}

// Clusters of n_split CTAs that can be resident at once (the occupancy
// query, once per context); 0 if none or unknown.
template <int HD, bool LW>
int tc_max_clusters(int n_split) {
  static ContextCache<int> cache[kMaxKeySplits + 1];
  int v = 0;
  if (!per_context(cache[n_split], &v, [n_split](int* out) {
        cudaLaunchAttribute attr[1];
        const cudaLaunchConfig_t cfg = tc_config<HD>(dim3(1, 1, n_split), n_split, nullptr, attr);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, (const void*)chunk_attn_tc<HD, LW>, &cfg) != cudaSuccess)
          return false;
        *out = n;
        return true;
      }))
    return 0;
  return v;
}

// Key splits per (row tile, KV head) (choose_key_splits), with the clusters
// that can be resident taken from the occupancy query.
template <int HD, bool LW>
int tc_key_splits(long long base, int n_all) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    (void)cudaGetLastError();
    return 1;
  }
  return choose_key_splits(base, n_all, sms, [](int ns) { return tc_max_clusters<HD, LW>(ns); });
}

// One CTA per (128 query rows, KV head, key split): 224 threads at head_dim
// 64 and 128, 256 at 256.
template <int HD, bool LW>
cudaError_t launch_tc_kernel(const ChunkArgs& a, cudaStream_t s) {
  using Lay = tcc::TcLayout<HD>;
  static ContextCache<int> limit_set;
  int done = 0;
  if (!per_context(limit_set, &done, [](int* v) {
        *v = 1;
        return cudaFuncSetAttribute(chunk_attn_tc<HD, LW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Lay::SMEM) == cudaSuccess;
      }))
    return cudaErrorInvalidConfiguration;
  ChunkMaps maps;
  memset(&maps, 0, sizeof(maps));
  const long long rows = (long long)a.n_kv * a.P;
  for (int sp = 0; sp < Lay::NSP; ++sp) {
    if (!make_span_map(&maps.k[sp], a.k16, sp, rows, HD * 2, Lay::BN) ||
        !make_span_map(&maps.v[sp], a.v16, sp, rows, HD * 2, Lay::BN))
      return cudaErrorInvalidValue;
  }
  const long long row_tiles = ((long long)a.T * a.G + tcc::BM - 1) / tcc::BM;
  if (row_tiles > 0x7fffffffLL || a.n_kv > 65535) return cudaErrorInvalidValue;
  const int n_split = tc_key_splits<HD, LW>(row_tiles * a.n_kv, (a.P + Lay::BN - 1) / Lay::BN);
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      tc_config<HD>(dim3((unsigned)row_tiles, (unsigned)a.n_kv, (unsigned)n_split), n_split, s, attr);
  return cudaLaunchKernelEx(&cfg, chunk_attn_tc<HD, LW>, maps, a);
}

template <int HD>
cudaError_t launch_tc(const ChunkArgs& a, cudaStream_t s) {
  return a.extra_tx != 0 ? launch_tc_kernel<HD, true>(a, s) : launch_tc_kernel<HD, false>(a, s);
}

}  // namespace

cudaError_t launch_chunk_attn(int hd, const ChunkArgs& a, cudaStream_t s) {
  switch (hd) {
    case 64: return launch_tc<64>(a, s);
    case 128: return launch_tc<128>(a, s);
    case 256: return launch_tc<256>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq

// kvq_decode_mma.cu -- split-K decode attention on tensor cores, fed by TMA.
//
// The partial kernel of the split-K decode (#3084 qwen35: FP16 K/V cache by
// default, int8 with --kv-q8, "What changed" and "Extra Notes": k_attn_part
// templated on the cache format, read by the decode of the next token).  One
// CTA of 4 warps per (split, KV head, sequence):
//
//   copies      the split's cells stream through a ring of STAGES
//               shared-memory stages of 64 cells: K and V codes by TMA
//               tensor copies (cp.async.bulk.tensor, 128-byte swizzle,
//               straight from the paged pool through the block table), the
//               scales by bulk copies; an mbarrier per stage counts the
//               bytes in.  Thread 0 issues the first stages; after that the
//               warp that releases a stage last (a shared-memory counter)
//               issues its refill.
//   q.k         each warp owns 16 cells of every stage.  S^T = K . Q^T is a
//               16-cell x 8-row mma.sync.m16n8k16 per 16 dims.  int8 K
//               enters as the exact fp16 value 1152 + code, and 1152 * sum(q)
//               per 64-dim group is taken off through the accumulator's
//               starting value; the per-64-dim scales multiply the group
//               partial dot products.
//   softmax     online, in the log2 domain, with a lazily raised reference
//               maximum.
//   p.v         O^T += V^T . P^T, another m16n8k16 per 16 dims; int8 V is
//               widened to fp16 exactly in registers and the V scales are
//               folded into P per group.  K8V4 (#711 kv: --kv k8v4 streams
//               with --kv-resident, "What"): K as int8; V's 4-bit codes
//               widen exactly to code - 8, its per-32 scales fold into P,
//               and each split's merged partial is rotated back
//               (Walsh-Hadamard, / HD) before it is written.
//
// q and p enter the tensor cores as fp16 hi + lo pairs (about 22 significant
// bits), K and V as exact fp16 values.  The copies carry an evict-first L2
// policy: the cache is read once per call.
//
// The CTA's 4 warps merge their states through shared memory into one
// partial (o, m, l) per row of the split; the combine kernel below merges
// the partials of every split.  Masked cells (beyond the context, beyond the causal limit of a
// verify-window row, or in a block whose id is out of range) get logit -inf
// and contribute exact zeros.  Every mbarrier wait is bounded: a wait that
// runs out marks the partial as NaN (the combine passes NaN to the output)
// and thread 0 still waits, bounded, for the CTA's copies before the CTA
// exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include <string.h>

#include <mutex>

#include "kvq_internal.cuh"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = kConsumerWarps * 32;  // thread 0 also issues the copies
constexpr int kTC = 64;                      // cells per pipeline stage (a piece index is
                                             // split by shifts: 64 = 2^6)
constexpr int kCellsPerWarp = kTC / kConsumerWarps;
constexpr float kTau = 8.0f;                 // lazy rescale threshold (log2 units)
constexpr unsigned kFull = 0xffffffffu;

template <int FMT, int HD, int NT>
struct Cfg {
  static constexpr bool KI8 = FMT != KVQ_F16;            // K as int8 codes + scales
  static constexpr bool V4 = FMT == KVQ_K8V4;            // V as rotated 4-bit codes
  static constexpr int ESZ = FMT == KVQ_F16 ? 2 : 1;
  static constexpr int ROWB = HD * ESZ;                  // K code bytes per cell row
  static constexpr int SWB = ROWB < 128 ? ROWB : 128;    // swizzle span (64 or 128 B)
  static constexpr int NCH = ROWB / SWB;                 // swizzle spans per row
  static constexpr int NG = HD / kGroup;
  static constexpr int VROWB = V4 ? HD / 2 : ROWB;       // V code bytes per cell row
  static constexpr int VSWB = VROWB < 128 ? VROWB : 128; // (32, 64 or 128 B)
  static constexpr int VNCH = VROWB / VSWB;
  static constexpr int VNS = V4 ? HD / kQ4Block : NG;    // V scales per cell row
  static constexpr int TILE_B = kTC * ROWB;              // K codes of a stage
  static constexpr int VTILE_B = kTC * VROWB;            // V codes of a stage
  static constexpr int KSCALE_B = KI8 ? kTC * NG * 2 : 0;
  static constexpr int VSCALE_B = KI8 ? kTC * VNS * 2 : 0;
  static constexpr int SC_STAGE_B = KSCALE_B + VSCALE_B;
  // A stage holds the K and V code tiles (each a whole number of 1 KB
  // swizzle atoms); the scales of all stages live in a region of their
  // own so no stage is padded.
  static constexpr int STAGE_B = TILE_B + VTILE_B;
  // Three stages per CTA (one landing while two are read) and as many
  // 4-warp CTAs per SM as the 227 KB allow keep about 100 KB or more of
  // copies in flight per SM.
  // (the merge at the end reuses the stages for 4 warp slabs of RP x HD
  // fp32, which takes a fourth stage for 32-row int8 HD 64 tiles)
  static constexpr int SLAB_B = kConsumerWarps * NT * 8 * HD * 4;
  static constexpr int STAGES = (SLAB_B + STAGE_B - 1) / STAGE_B > 3 ? (SLAB_B + STAGE_B - 1) / STAGE_B : 3;
  static constexpr int OFF_V = TILE_B;
  static constexpr int SMEM_SC = STAGES * STAGE_B;  // [STAGES]{K [64][NG], V [64][VNS]} fp16
  // q as fp16 hi / lo rows, padded by 16 bytes so ldmatrix rows hit distinct banks
  static constexpr int QROW = HD * 2 + 16;
  static constexpr int QBYTES_MAX = 2 * NT * 8 * QROW;   // hi and lo, NT*8 padded rows
  static constexpr int SMEM_Q = SMEM_SC + STAGES * SC_STAGE_B;
  // int8: per (padded row, 64-dim group, 32-dim half) 1152 * sum of q (hi + lo)
  static constexpr int SMEM_QC = SMEM_Q + (QBYTES_MAX + 15) / 16 * 16;
  static constexpr int QC_BYTES = KI8 ? (NT * 8 * NG * 2 * 4 + 15) / 16 * 16 : 0;
  // per-warp row maxima and sums for the merge at the end: [4][RP][2] fp32
  static constexpr int SMEM_WML = SMEM_QC + QC_BYTES;
  static constexpr int SMEM_BAR = SMEM_WML + kConsumerWarps * NT * 8 * 2 * 4;
  // block ids of the split's pieces, staged once so any warp can issue a refill
  static constexpr int ROWS_CAP = 128;
  static constexpr int SMEM_REL = SMEM_BAR + STAGES * 8;        // release counters [STAGES]
  static constexpr int SMEM_BLK = SMEM_REL + 16 * 4;            // block ids [ROWS_CAP]
  static constexpr int SMEM = SMEM_BLK + ROWS_CAP * 4 + 1024 /*align*/;
  static constexpr int FIT = (228 * 1024) / (SMEM + 1024);  // 1 KB reserved per CTA
  // 32-row tiles (NT 4) hold 4x the accumulators: at most 3 CTAs (168
  // registers a thread) so they do not spill
  // (K8V4's 16-row tiles, whose smaller stages would fit 4, likewise)
  static constexpr int FIT_R = (NT >= 4 || (V4 && NT >= 2)) ? (FIT < 3 ? FIT : 3) : FIT;
  static constexpr int MIN_CTAS = FIT_R >= 4 ? 4 : (FIT_R >= 3 ? 3 : (FIT_R >= 2 ? 2 : 1));
  static_assert(STAGES * STAGE_B >= SLAB_B, "merge slabs fit in the stages");
  // the SM's 228 KB hold MIN_CTAS of these CTAs (1 KB of each is reserved)
  static_assert(MIN_CTAS * (SMEM + 1024) <= 228 * 1024, "CTAs per SM fit the shared memory");
};

// One 2D tensor map per SWB-byte span of a cell row: [rows][SWB], row
// stride = the row's bytes.  A piece of pc cells lands as [span][cell][SWB].
struct TmaMaps {
  CUtensorMap k[4];
  CUtensorMap v[4];
};

// int8 -> fp16, exactly: with u = c ^ 0x80 (= c + 128 as an unsigned byte),
// the fp16 bit pattern 0x6400 | u is 1024 + u, and (1024 + u) - 1152 = c.
constexpr uint32_t kMagic = 0x64646464u;
constexpr uint32_t kBias = 0x64806480u;  // fp16 1152 in both halves

// Swizzled shared-memory byte offset of logical byte `b` of cell `c` (0..63)
// in a K or V tile laid out [span][cell][SWB]: every TMA box (one piece of
// cells, one span) is placed at its [span][first cell] slot, so the layout
// and the swizzle (XOR of the 16-byte chunk with the line index mod 8 or 4)
// do not depend on the block size.
__device__ __forceinline__ uint32_t swz_off(int c, int b, int sw) {
  const uint32_t off = ((uint32_t)(b / sw) * kTC + (uint32_t)c) * sw + (uint32_t)(b % sw);
  // 128-byte swizzle: chunk bits [4:6] ^= address bits [7:9]; 64-byte:
  // [4:5] ^= [7:8]; 32-byte: [4] ^= [7]
  return off ^ (((off >> 7) & (uint32_t)(sw / 16 - 1)) << 4);
}

template <int FMT, int HD>
__device__ __forceinline__ uint32_t tile_off(int c, int b) {
  return swz_off(c, b, Cfg<FMT, HD, 1>::SWB);
}

// r / G for a query row index r (r < 32 <= 2^32 / G): a multiply by the
// host's ceil(2^32 / G) instead of a division by a run-time value, which
// sat on the path to each CTA's first copy (8 q loads a thread, each with
// a row index to divide)
__device__ __forceinline__ int div_g(const DecodeArgs& a, int r) {
  return (int)(((unsigned long long)(unsigned)r * a.g_magic) >> 32);
}

__device__ __forceinline__ int clamp_len_mma(int L, const DecodeArgs& a) {
  const long long cap_table = (long long)a.max_blocks << a.pool.bs_log2;
  const long long cap_plan = (long long)a.nsplit * a.split_cells;
  const long long cap = cap_table < cap_plan ? cap_table : cap_plan;
  return L < 0 ? 0 : (int)((long long)L < cap ? L : cap);
}


// Block id of cell c (-1 past the end).  Loaded a tile ahead of its use and
// only tested when used, so the load latency stays hidden.
__device__ __forceinline__ int block_of(const DecodeArgs& a, const int32_t* bt, int c, int c_end) {
  return c < c_end ? __ldg(bt + (c >> a.pool.bs_log2)) : -1;
}

// Work item of CTA c.  The grid is one CTA per possible (sequence, KV head,
// split); the items that hold cells are numbered so that every full-length
// split comes first (in sequence, split, KV head order) and the last,
// shorter split of each sequence after them.  CTAs are dispatched roughly in
// index order, so the short splits fill the tail of the launch instead of
// full-length splits starting last.  Every warp computes this itself, a
// warp-wide scan over 32 sequences at a time.  Returns false past the end.
__device__ __forceinline__ bool item_of(const DecodeArgs& a, int c, int& b, int& kvh, int& split) {
  const int lane = threadIdx.x & 31;
  const int S = a.split_cells, nkv = a.pool.n_kv;
  for (int pass = 0; pass < 2; ++pass) {   // 0: full splits, 1: last partial splits
    for (int b0 = 0; b0 < a.n_seq; b0 += 32) {
      const int bb = b0 + lane;
      int n = 0, Lb = 0;
      if (bb < a.n_seq) {
        Lb = clamp_len_mma(__ldg(a.ctx_lens + bb), a);
        const int qs = (int)fdiv((unsigned)Lb, a.div_split);   // Lb / S (Lb >= 0)
        n = pass == 0 ? qs * nkv : (Lb - qs * S != 0 ? nkv : 0);
      }
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += y;
      }
      const int total = __shfl_sync(kFull, incl, 31);
      if (c < total) {
        const unsigned m = __ballot_sync(kFull, bb < a.n_seq && incl > c);
        const int src = __ffs(m) - 1;
        const int k = c - __shfl_sync(kFull, incl - n, src);
        const int Ls = __shfl_sync(kFull, Lb, src);
        b = b0 + src;
        if (pass == 0) {
          split = (int)fdiv((unsigned)k, a.div_nkv);
          kvh = k - split * nkv;
        } else {
          split = (int)fdiv((unsigned)Ls, a.div_split);
          kvh = k;
        }
        return true;
      }
      c -= total;
    }
  }
  return false;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// HL (at most 4 query rows, NT = 1): the MMA's 8 columns carry the hi
// parts of q (and of p) in columns 0-3 and the lo parts in columns 4-7, so
// each k-step of q.k and each m-tile of p.v takes one MMA instead of two;
// the hi and lo sums meet by one shuffle (lanes t and t ^ 2): per tile for
// the logits, once per split for the output.  q's fragments stay in
// registers.
template <int FMT, int HD, int NT, bool HL>
__global__ void __launch_bounds__(kThreads, Cfg<FMT, HD, NT>::MIN_CTAS)
    decode_mma(const __grid_constant__ TmaMaps maps, DecodeArgs a) {
  static_assert(!HL || NT == 1, "hi/lo columns need a single 8-column row tile");
  using C = Cfg<FMT, HD, NT>;
  constexpr int KS = HD / 16;   // k-steps of q.k, and m-tiles of p.v
  constexpr int RP = NT * 8;    // padded rows
  constexpr int MAXP = kTC / 16;
  constexpr float kNegInf = -INFINITY;
  constexpr float kMStart = -1e30f;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t qbase = sbase + C::SMEM_Q;                 // q hi rows, then lo rows
  const uint32_t bar_full = sbase + C::SMEM_BAR;
  int* s_rel = reinterpret_cast<int*>(smem + C::SMEM_REL);
  int* s_blk = reinterpret_cast<int*>(smem + C::SMEM_BLK);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Launched as a programmatic dependent of the previous kernel on the
  // stream: nothing it may have written is read before this wait.
  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.k[0])) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.v[0])) : "memory");
    // One sequence: while the previous kernel finishes, the first two tiles
    // of this CTA's split are brought into L2.  Only a hint: the block
    // ids read here may still change before the wait below (the copies
    // read them again after the wait), and a prefetch of the wrong rows
    // costs bandwidth, nothing else.
    if (a.n_seq == 1 && a.n_rt == 1) {
      const int split0 = (int)fdiv(blockIdx.x, a.div_nkv), kvh0 = (int)blockIdx.x - split0 * a.pool.n_kv;
      const int c0 = split0 * a.split_cells;
      const int pcl = a.pool.bs_log2 < 6 ? a.pool.bs_log2 : 6;
      const int cap = clamp_len_mma(INT_MAX, a);   // cells the table row can address
      if (c0 < cap) {
        constexpr int kPrefetchTiles = 2;
        for (int p = 0; p < kPrefetchTiles * (kTC >> pcl) && (p << pcl) < a.split_cells && c0 + (p << pcl) < cap;
             ++p) {
          // read at L2 (no L1 line: the reads after the wait must not
          // find a copy taken before the previous kernel's writes)
          const int blk = __ldcg(a.block_table + ((c0 + (p << pcl)) >> a.pool.bs_log2));
          if (blk < 0 || blk >= a.pool.n_blocks) continue;
          const size_t row =
              ((size_t)blk * a.pool.n_kv + kvh0) * (1u << a.pool.bs_log2) + ((c0 + (p << pcl)) & ((1 << a.pool.bs_log2) - 1));
          const uint32_t n = 1u << pcl;
          prefetch_l2(static_cast<const char*>(a.pool.k) + row * C::ROWB, n * C::ROWB);
          prefetch_l2(static_cast<const char*>(a.pool.v) + row * C::VROWB, n * C::VROWB);
          if constexpr (C::KI8) {
            prefetch_l2(a.pool.ks + row * C::NG, n * C::NG * 2);
            prefetch_l2(a.pool.vs + row * C::VNS, n * C::VNS * 2);
          }
        }
      }
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // One sequence: CTA c is split c / n_kv of KV head c % n_kv whatever the
  // context length (the item order below reduces to that), so the block
  // ids and the first copies need not wait for the length, which is only
  // read after them; a split that turns out to lie past the context marks
  // its slots empty.  A batch: CTAs past the last item (splits beyond a
  // sequence's context) have nothing to do; the combine kernel reads only
  // the slots of live splits.
  // Row tiles: a work item's R query rows are cut into tiles of a.RT rows
  // (a verify window wider than one CTA's accumulators), one CTA each; the
  // CTAs of an item are neighbours in the grid, so all but the first find
  // the item's K/V tiles in L2.
  const int item = (int)fdiv(blockIdx.x, a.div_nrt);
  const int r0 = ((int)blockIdx.x - item * a.n_rt) * a.RT;  // first query row of this CTA
  const int Rc = min(a.RT, a.R - r0);                         // and its row count
  int b, kvh, split;
  int L_raw = 0;
  const bool single = a.n_seq == 1;
  if (single) {
    b = 0;
    split = (int)fdiv((unsigned)item, a.div_nkv);
    kvh = item - split * a.pool.n_kv;
    L_raw = __ldg(a.ctx_lens);
  } else {
    if (!item_of(a, item, b, kvh, split)) return;
    L_raw = __ldg(a.ctx_lens + b);
  }
  const int c_begin = split * a.split_cells;
  // until the length is known (one sequence), copies stay inside the split
  // and the block table
  int c_end = min(clamp_len_mma(single ? INT_MAX : L_raw, a), c_begin + a.split_cells);
  int n_tiles = (c_end - c_begin + kTC - 1) / kTC;
  const int n_first = n_tiles < C::STAGES ? n_tiles : C::STAGES;   // tiles of the first wave
  const int pc_log2 = a.pool.bs_log2 < 6 ? a.pool.bs_log2 : 6;  // cells per TMA piece
  const int n_pieces = kTC >> pc_log2;
  const int32_t* bt = a.block_table + (size_t)b * a.max_blocks;
  const bool producer = threadIdx.x == 0;
  // the cache is read once per call: its lines leave L2 first
  const uint64_t pol = l2_evict_first_policy();
  // Let the combine grid be scheduled as soon as SMs free up; it still waits
  // (griddepcontrol.wait) for this whole grid to finish before reading.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Copies of a stage are issued by whichever warp releases the stage last
  // (a shared-memory counter per stage), so no warp ever blocks waiting for
  // the others.  The block id of every piece of the split is staged in
  // shared memory once (when it fits), so an issuing warp needs no global
  // load on that path.
  const int n_entries = n_tiles * n_pieces;
  const bool blk_in_smem = n_entries <= C::ROWS_CAP;
  auto piece_blk = [&](int it, int p, bool from_smem) -> int {
    return from_smem ? s_blk[it * n_pieces + p]
                     : block_of(a, bt, c_begin + it * kTC + (p << pc_log2), c_end);
  };
  // block ids of the pieces of tile it
  auto tile_blks = [&](int it, bool from_smem, int (&blk)[MAXP]) {
#pragma unroll
    for (int p = 0; p < MAXP; ++p) blk[p] = p < n_pieces ? piece_blk(it, p, from_smem) : -1;
  };
  auto issue = [&](int it, const int (&blks)[MAXP]) {
    const int s = it % C::STAGES;
    const int pc = 1 << pc_log2;
    const int bsz = 1 << a.pool.bs_log2;
    const int c0 = c_begin + it * kTC;
    int rows[MAXP];
    uint32_t bytes = 0;
#pragma unroll
    for (int p = 0; p < MAXP; ++p) {
      const int blk = blks[p];
      const int c = c0 + (p << pc_log2);
      rows[p] = (p < n_pieces && blk >= 0 && blk < a.pool.n_blocks)
                    ? (blk * a.pool.n_kv + kvh) * bsz + (c & (bsz - 1))
                    : -1;
      if (rows[p] >= 0) bytes += (uint32_t)pc * (C::ROWB + C::VROWB + (C::KI8 ? (C::NG + C::VNS) * 2 : 0));
    }
    const uint32_t full = bar_full + 8 * s;
    mbar_expect_tx(full, bytes + a.extra_tx);
    const uint32_t st = sbase + s * C::STAGE_B;
    for (int p = 0; p < n_pieces; ++p) {
      const int row = rows[p];
      if (row < 0) continue;
#pragma unroll
      for (int sp = 0; sp < C::NCH; ++sp) {
        const uint32_t so = (uint32_t)(sp * kTC + (p << pc_log2)) * C::SWB;
        tma_load_2d_hint(st + so, &maps.k[sp], 0, row, full, pol);
      }
#pragma unroll
      for (int sp = 0; sp < C::VNCH; ++sp) {
        const uint32_t so = (uint32_t)(sp * kTC + (p << pc_log2)) * C::VSWB;
        tma_load_2d_hint(st + C::OFF_V + so, &maps.v[sp], 0, row, full, pol);
      }
      if constexpr (C::KI8) {
        const uint32_t sbk = (uint32_t)pc * C::NG * 2, sbv = (uint32_t)pc * C::VNS * 2;
        const uint32_t sc = sbase + C::SMEM_SC + (uint32_t)s * C::SC_STAGE_B;
        bulk_load_hint(sc + (uint32_t)p * sbk, a.pool.ks + (size_t)row * C::NG, sbk, full, pol);
        bulk_load_hint(sc + C::KSCALE_B + (uint32_t)p * sbv, a.pool.vs + (size_t)row * C::VNS, sbv, full, pol);
      }
    }
  };

  // Prologue.  Every small load (q, the split's block ids) is issued first,
  // into registers; only then does thread 0 start the first stages' bulk
  // copies.  Issued the other way round, these few latency-critical loads
  // would queue behind tens of megabytes of copies from all CTAs.
  //
  // q * sm_scale * log2(e) goes to shared memory as fp16 hi + lo, rows
  // [RP][HD] in k order: FP16 uses the natural dim order; int8 permutes each
  // 16-wide k-step ks so that k = 2t + e -> dim 16 ks + 4 t + e and
  // k = 2t + 8 + e -> that + 2 (t = k-pair lane): a lane's ldmatrix word
  // holds the 4 code bytes of dims 16 ks + 4t .. + 3.
  constexpr int QPT = (RP * HD + kThreads - 1) / kThreads;  // q values per thread
  constexpr int BPT = (C::ROWS_CAP + kThreads - 1) / kThreads;
  float qv[QPT];
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = threadIdx.x + u * kThreads;
    qv[u] = 0.f;
    if (i < RP * HD) {
      const int r = i / HD, k = i - r * HD;
      int dim = k;
      if constexpr (C::KI8) {
        const int ks = k >> 4, kq = k & 15;
        const int tt = (kq & 7) >> 1, e = kq & 1, hi8 = kq >> 3;
        dim = 16 * ks + 4 * tt + 2 * hi8 + e;
      }
      if (r < Rc) {
        const int w = div_g(a, r0 + r), gg = r0 + r - w * a.G;
        qv[u] = __ldg(a.q + (((size_t)b * a.W + w) * a.n_q + (size_t)kvh * a.G + gg) * HD + dim);
      }
    }
  }
  int bv[BPT];
#pragma unroll
  for (int u = 0; u < BPT; ++u) {
    const int i = threadIdx.x + u * kThreads;
    bv[u] = (blk_in_smem && i < n_entries)
                ? block_of(a, bt, c_begin + (i >> (6 - pc_log2)) * kTC + ((i & (n_pieces - 1)) << pc_log2), c_end)
                : -1;
  }
  bool lost = false;
  if (producer) {
    // the block ids of every first-wave piece are loaded together, before
    // the first copy is issued
    int fb[C::STAGES][MAXP];
#pragma unroll
    for (int it = 0; it < C::STAGES; ++it) tile_blks(it, false, fb[it]);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      s_rel[s] = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the first tile now; the rest of the first wave after the barrier
    // below, so that on every SM each CTA's first tile is queued for the
    // copy engine ahead of the other tiles of the wave
    if (n_first > 0) issue(0, fb[0]);
  }
  {
    unsigned char* qs = smem + C::SMEM_Q;
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
      const int i = threadIdx.x + u * kThreads;
      if (i < RP * HD && (!HL || i / HD < 4)) {
        const int r = i / HD, k = i - r * HD;
        const float x = qv[u] * a.qscale;
        const __half h = __float2half_rn(x);
        const __half lo = __float2half_rn(x - __half2float(h));
        *reinterpret_cast<__half*>(qs + r * C::QROW + k * 2) = h;
        *reinterpret_cast<__half*>(qs + (HL ? 4 + r : RP + r) * C::QROW + k * 2) = lo;
        if constexpr (C::KI8) {
          // The 32 lanes of a warp hold 32 consecutive k of one row and one
          // 64-dim group (RP * HD is a multiple of 128): their sum of q,
          // times 1152, fills the (row, group, half) slot of the int8 bias.
          float v = __half2float(h) + __half2float(lo);
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
          if (lane == 0)
            reinterpret_cast<float*>(smem + C::SMEM_QC)[(r * C::NG + k / 64) * 2 + ((k >> 5) & 1)] =
                1152.0f * v;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < BPT; ++u) {
      const int i = threadIdx.x + u * kThreads;
      if (blk_in_smem && i < n_entries) s_blk[i] = bv[u];
    }
  }
  __syncthreads();
  const int L = clamp_len_mma(L_raw, a);
  if (single) {
    c_end = min(L, c_begin + a.split_cells);
    n_tiles = c_end > c_begin ? (c_end - c_begin + kTC - 1) / kTC : 0;
    if (n_tiles == 0) {
      // a split past the context: its slots tell the combine "no cells"
      if (producer && n_first > 0) (void)mbar_wait(bar_full, 0, a.wait_limit);
      const size_t slot0 = (((size_t)b * a.pool.n_kv + kvh) * a.nsplit + split) * a.R;
      if (threadIdx.x < a.R)
        *reinterpret_cast<float2*>(a.ws_ml + (slot0 + threadIdx.x) * 2) = make_float2(-INFINITY, 0.f);
      return;
    }
  }
  if (producer) {
    for (int it = 1; it < n_first; ++it) {
      int nb[MAXP];
      tile_blks(it, blk_in_smem, nb);
      issue(it, nb);
    }
  }

  // ---------------- consumer setup ----------------
  const int g = lane >> 2, t = lane & 3;

  // int8 K enters the MMA as fp16 (1152 + code) (no subtraction per
  // element); the 1152 * sum(q) of each (row, 64-dim group) is taken off
  // once, as the starting value of that group's hi accumulator.
  float qcorr[C::KI8 ? C::NG : 1][NT][2];
  if constexpr (C::KI8) {
    const float* s_qc = reinterpret_cast<const float*>(smem + C::SMEM_QC);
#pragma unroll
    for (int gq = 0; gq < C::NG; ++gq)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int i = ((nt * 8 + 2 * t + j) * C::NG + gq) * 2;
          // (HL: the lo columns 4-7 start at 0; the hi ones carry the whole
          // correction, the two meet in the logits)
          qcorr[gq][nt][j] = (HL && t >= 2) ? 0.f : -(s_qc[i] + s_qc[i + 1]);
        }
  }

  // ldmatrix lane addressing of q: matrix lane>>3 = {hi k0-7, hi k8-15, lo
  // k0-7, lo k8-15}, row lane&7.
  const uint32_t q_lane = qbase + (uint32_t)((lane >> 4) * RP + (lane & 7)) * C::QROW +
                          (uint32_t)((lane >> 3) & 1) * 16;
  // HL: the B fragments of every k-step (rows 0-3 hi, 4-7 lo), kept in
  // registers; one ldmatrix x4 covers two k-steps
  uint32_t qreg[HL ? KS : 1][2];
  if constexpr (HL) {
    const uint32_t ql = qbase + (uint32_t)(lane & 7) * C::QROW + (uint32_t)(lane >> 3) * 16;
#pragma unroll
    for (int ks = 0; ks < KS; ks += 2) {
      uint32_t r4[4];
      ldsm_x4(r4, ql + ks * 32);
      qreg[ks][0] = r4[0];
      qreg[ks][1] = r4[1];
      qreg[ks + 1][0] = r4[2];
      qreg[ks + 1][1] = r4[3];
    }
  }

  // Last visible cell of each of this thread's rows (the verify window's
  // causal limit), or -1 for padding rows.
  // the query row of this thread's column j of row tile nt (HL: lanes t
  // and t ^ 2 hold the same rows, hi and lo halves)
  auto row_of = [&](int nt, int j) -> int { return HL ? 2 * (t & 1) + j : nt * 8 + 2 * t + j; };
  int row_last[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = row_of(nt, j);
      row_last[nt][j] = r < Rc ? L - a.W + div_g(a, r0 + r) : -1;
    }

  int row_last_min = INT_MAX;  // smallest causal limit among this thread's real rows
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (row_of(nt, j) < Rc) row_last_min = min(row_last_min, row_last[nt][j]);

  float m[NT][2], l[NT][2];
  float o[KS][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // a finite start, so p needs no "no maximum yet" test: the first tile
    // with a visible cell always raises it
    m[nt][0] = m[nt][1] = kMStart;
    l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
  }

  const int cl = warp * kCellsPerWarp;  // first cell of this warp's slice in a stage
  auto slice_blk = [&](int it) -> int {
    if (it >= n_tiles) return -1;
    if (blk_in_smem) return c_begin + it * kTC + cl < c_end ? s_blk[it * n_pieces + (cl >> pc_log2)] : -1;
    return block_of(a, bt, c_begin + it * kTC + cl, c_end);
  };
  auto slice_nvalid = [&](int it, int blk) -> int {
    return (blk >= 0 && blk < a.pool.n_blocks) ? min(kCellsPerWarp, c_end - (c_begin + it * kTC + cl)) : 0;
  };

  // Swizzled shared-memory addresses.  With a 128-byte swizzle the XOR term
  // of every address this thread reads splits into a per-thread constant and
  // a compile-time part, so a few base registers replace the full
  // computation per load (the spans of a row are whole 64-cell x 128-byte
  // blocks, reached by immediate offsets).
  //
  // ldmatrix x4 lane addressing: matrix mi = lane >> 3 reads row rr = lane & 7.
  // kx: matrices (cells +0, chunk 2k), (cells +8, chunk 2k), (cells +0,
  // chunk 2k+1), (cells +8, chunk 2k+1) of the k-th 32-byte step of a row --
  // K for q.k in both formats and, as byte pairs, int8 V for p.v.  vx (FP16
  // V^T): (cells +0, chunk 2k), (+0, 2k+1), (+8, 2k), (+8, 2k+1).
  constexpr uint32_t kSpanB = kTC * 128;
  uint32_t kx[4], vx[4];
  {
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t ck = (uint32_t)(cl + ((mi & 1) << 3) + rr), cv = (uint32_t)(cl + ((mi >> 1) << 3) + rr);
    if constexpr (C::SWB == 128) {
      const uint32_t xk = ((uint32_t)(mi >> 1) << 4) ^ ((uint32_t)rr << 4);
      const uint32_t xv = ((uint32_t)(mi & 1) << 4) ^ ((uint32_t)rr << 4);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        kx[k] = ck * 128 + (xk ^ (32u * k));
        vx[k] = C::OFF_V + cv * 128 + (xv ^ (32u * k));
      }
    } else {  // 64-byte rows (int8, HD 64): two 32-byte steps
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        kx[k] = tile_off<FMT, HD>((int)ck, (32 * k + 16 * (mi >> 1)) & (C::ROWB - 1));
        vx[k] = 0;
      }
    }
  }
  // K8V4 V: the same matrix order over 16-byte chunks of the nibble rows
  // (chunk = one 32-dim block), in the V tile's own swizzle span.
  uint32_t vq[C::V4 ? C::VROWB / 32 : 1];
  if constexpr (C::V4) {
    const int mi = lane >> 3, rr = lane & 7;
    const int ck = cl + ((mi & 1) << 3) + rr;
#pragma unroll
    for (int k = 0; k < C::VROWB / 32; ++k) vq[k] = C::OFF_V + swz_off(ck, 32 * k + 16 * (mi >> 1), C::VSWB);
  }
  // shared-memory offset of the k-th 32-byte step of the kx row set
  auto kstep = [&](int k) -> uint32_t {
    if constexpr (C::SWB == 128) return kx[k & 3] + (uint32_t)(k >> 2) * kSpanB;
    else return kx[k & 1];
  };

  // q . k of one stage for this warp's 16 cells -> z (log2-domain logits)
  auto qk = [&](int s, float (&z)[NT][4]) {
    const uint32_t st = sbase + s * C::STAGE_B;
  // ---------------- S^T = K . Q^T (four independent accumulators) ----------------
  if constexpr (FMT == KVQ_F16 && HL) {
    float acc[2][4];  // alternate k-steps, two independent chains
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t af[4];
      ldsm_x4(af, st + kx[ks & 3] + (uint32_t)(ks >> 2) * kSpanB);
      if (ks < 2) mma16816_zc(acc[ks & 1], af, qreg[ks][0], qreg[ks][1]);
      else mma16816(acc[ks & 1], af, qreg[ks][0], qreg[ks][1]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float v = acc[0][k] + acc[1][k];
      z[0][k] = v + __shfl_xor_sync(kFull, v, 2);  // hi columns + lo columns
    }
  } else if constexpr (FMT == KVQ_F16) {
    float acc[4][NT][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t af[4];
      ldsm_x4(af, st + kx[ks & 3] + (uint32_t)(ks >> 2) * kSpanB);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint32_t qf[4];
        ldsm_x4(qf, q_lane + (uint32_t)(nt * 8) * C::QROW + ks * 32);
        if (ks < 2) {
          mma16816_zc(acc[(ks & 1) * 2 + 0][nt], af, qf[0], qf[1]);
          mma16816_zc(acc[(ks & 1) * 2 + 1][nt], af, qf[2], qf[3]);
        } else {
          mma16816(acc[(ks & 1) * 2 + 0][nt], af, qf[0], qf[1]);
          mma16816(acc[(ks & 1) * 2 + 1][nt], af, qf[2], qf[3]);
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        z[nt][k] = (acc[0][nt][k] + acc[2][nt][k]) + (acc[1][nt][k] + acc[3][nt][k]);
  } else {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) z[nt][0] = z[nt][1] = z[nt][2] = z[nt][3] = 0.f;
    const unsigned short* ksc = reinterpret_cast<const unsigned short*>(smem + C::SMEM_SC + s * C::SC_STAGE_B);
#pragma unroll
    for (int gq = 0; gq < C::NG; ++gq) {
      // words: [k-step kk][cells +0 | +8], each the 4 code bytes of dims
      // 16 (4 gq + kk) + 4t .. + 3 of cell g (or g + 8)
      uint32_t w[4][2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r[4];
        ldsm_x4(r, st + kstep(2 * gq + h));
        w[2 * h][0] = r[0] ^ 0x80808080u;
        w[2 * h][1] = r[1] ^ 0x80808080u;
        w[2 * h + 1][0] = r[2] ^ 0x80808080u;
        w[2 * h + 1][1] = r[3] ^ 0x80808080u;
      }
      float acc[2][NT][4];  // hi chain (starts at -1152 sum q), lo chain
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        acc[0][nt][0] = acc[0][nt][2] = qcorr[gq][nt][0];
        acc[0][nt][1] = acc[0][nt][3] = qcorr[gq][nt][1];
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t af[4];  // fp16 1152 + code, exact
        af[0] = prmt(w[kk][0], kMagic, 0x4140u);
        af[2] = prmt(w[kk][0], kMagic, 0x4342u);
        af[1] = prmt(w[kk][1], kMagic, 0x4140u);
        af[3] = prmt(w[kk][1], kMagic, 0x4342u);
        if constexpr (HL) {
          // one chain: columns 0-3 hi (start at -1152 sum q), 4-7 lo (at 0)
          mma16816(acc[0][0], af, qreg[gq * 4 + kk][0], qreg[gq * 4 + kk][1]);
        } else {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            uint32_t qf[4];
            ldsm_x4(qf, q_lane + (uint32_t)(nt * 8) * C::QROW + (gq * 4 + kk) * 32);
            mma16816(acc[0][nt], af, qf[0], qf[1]);
            if (kk == 0) mma16816_zc(acc[1][nt], af, qf[2], qf[3]);
            else mma16816(acc[1][nt], af, qf[2], qf[3]);
          }
        }
      }
      const float s0 = __half2float(__ushort_as_half(ksc[(cl + g) * C::NG + gq]));
      const float s8 = __half2float(__ushort_as_half(ksc[(cl + g + 8) * C::NG + gq]));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if constexpr (HL) {
          z[nt][0] = fmaf(s0, acc[0][nt][0], z[nt][0]);
          z[nt][1] = fmaf(s0, acc[0][nt][1], z[nt][1]);
          z[nt][2] = fmaf(s8, acc[0][nt][2], z[nt][2]);
          z[nt][3] = fmaf(s8, acc[0][nt][3], z[nt][3]);
        } else {
          z[nt][0] = fmaf(s0, acc[0][nt][0] + acc[1][nt][0], z[nt][0]);
          z[nt][1] = fmaf(s0, acc[0][nt][1] + acc[1][nt][1], z[nt][1]);
          z[nt][2] = fmaf(s8, acc[0][nt][2] + acc[1][nt][2], z[nt][2]);
          z[nt][3] = fmaf(s8, acc[0][nt][3] + acc[1][nt][3], z[nt][3]);
        }
      }
    }
    if constexpr (HL) {
#pragma unroll
      for (int k = 0; k < 4; ++k) z[0][k] += __shfl_xor_sync(kFull, z[0][k], 2);  // hi + lo columns
    }
  }

  };

  // causal / length masks, online softmax -> p (rescales o when the maximum rises)
  auto softmax = [&](int nvalid, int cw0, float (&z)[NT][4], float (&p)[NT][4]) {
    // padding rows never reach the output, so only a short slice or a causal
    // limit inside it needs masks
    const bool need_mask = nvalid < kCellsPerWarp || row_last_min - cw0 < kCellsPerWarp - 1;
  // ---------------- masks and online softmax ----------------
  // A row's maximum over the slice (8 lanes) is needed only when the
  // reference maximum must rise; that happens only if some lane's own
  // maximum lies above it by more than kTau, so one warp vote decides
  // whether the shuffles run at all (the outcome is the same either way).
  // p is first computed against the current reference maximum, ahead of
  // the vote, so its exponentials need not wait for the branch; the rare
  // tile that raises the maximum computes p again.
  auto probs = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        p[nt][j] = fast_exp2(z[nt][j] - m[nt][j]);
        p[nt][2 + j] = fast_exp2(z[nt][2 + j] - m[nt][j]);
      }
  };
  float lmax[NT][2];
  bool rise = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (need_mask) {
        const int vis = min(nvalid - 1, row_last[nt][j] - cw0);  // last visible slice index
        if (g > vis) z[nt][j] = kNegInf;
        if (g + 8 > vis) z[nt][2 + j] = kNegInf;
      }
      lmax[nt][j] = fmaxf(z[nt][j], z[nt][2 + j]);
      rise |= lmax[nt][j] > m[nt][j] + kTau;  // also true for the first finite maximum
    }
  }
  probs();
  if (__any_sync(kFull, rise)) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float tmax = lmax[nt][j];
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 4));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
        if (tmax > m[nt][j] + kTau) {
          const float alpha = fast_exp2(m[nt][j] - tmax);  // 0 from the finite start
          m[nt][j] = tmax;
          l[nt][j] *= alpha;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            o[mt][nt][j] *= alpha;
            o[mt][nt][2 + j] *= alpha;
          }
        }
      }
    }
    probs();
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) l[nt][j] += p[nt][j] + p[nt][2 + j];

  };

  // o += V^T . P^T for one stage
  auto pv = [&](int s, int nvalid, const float (&p)[NT][4]) {
    const uint32_t st = sbase + s * C::STAGE_B;
  // ---------------- O^T += V^T . P^T ----------------
  if constexpr (FMT == KVQ_F16) {
    uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      uint32_t h01, l01, h23, l23;
      split_pair(p[nt][0], p[nt][1], h01, l01);
      split_pair(p[nt][2], p[nt][3], h23, l23);
      if constexpr (HL) {  // columns 0-3 hi, 4-7 lo
        bh[nt][0] = movmatrix_t(t >= 2 ? l01 : h01);
        bh[nt][1] = movmatrix_t(t >= 2 ? l23 : h23);
      } else {
        bh[nt][0] = movmatrix_t(h01);
        bh[nt][1] = movmatrix_t(h23);
        bl[nt][0] = movmatrix_t(l01);
        bl[nt][1] = movmatrix_t(l23);
      }
    }
    // V rows of cells past the valid ones may hold anything: zero them.
    const uint32_t mlo = (2 * t < nvalid ? 0xffffu : 0u) | (2 * t + 1 < nvalid ? 0xffff0000u : 0u);
    const uint32_t mhi =
        (2 * t + 8 < nvalid ? 0xffffu : 0u) | (2 * t + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t af[4];
      ldsm_x4_t(af, st + vx[mt & 3] + (uint32_t)(mt >> 2) * kSpanB);
      if (nvalid < kCellsPerWarp) {
        af[0] &= mlo;
        af[1] &= mlo;
        af[2] &= mhi;
        af[3] &= mhi;
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma16816(o[mt][nt], af, bh[nt][0], bh[nt][1]);
        if constexpr (!HL) mma16816(o[mt][nt], af, bl[nt][0], bl[nt][1]);
      }
    }
  } else if constexpr (C::V4) {
    // The fp16 scales of this thread's cells g and g + 8 (the rows of its
    // p fragments), every 32-dim block: one vector load per cell.
    constexpr int SWD = C::VNS / 2;
    const unsigned char* vsc = smem + C::SMEM_SC + s * C::SC_STAGE_B + C::KSCALE_B;
    uint32_t sw[2][SWD];
#pragma unroll
    for (int ci = 0; ci < 2; ++ci) {
      const unsigned char* src = vsc + (cl + g + 8 * ci) * (C::VNS * 2);
      if constexpr (SWD == 4) {
        const uint4 u = *reinterpret_cast<const uint4*>(src);
        sw[ci][0] = u.x;
        sw[ci][SWD > 1 ? 1 : 0] = u.y;
        sw[ci][SWD > 2 ? 2 : 0] = u.z;
        sw[ci][SWD > 3 ? 3 : 0] = u.w;
      } else if constexpr (SWD == 2) {
        const uint2 u = *reinterpret_cast<const uint2*>(src);
        sw[ci][0] = u.x;
        sw[ci][SWD > 1 ? 1 : 0] = u.y;
      } else {
        sw[ci][0] = *reinterpret_cast<const uint32_t*>(src);
      }
#pragma unroll
      for (int i = 0; i < SWD; ++i) sw[ci][i] = clamp_finite_h2(sw[ci][i]);
    }
    // One ldmatrix.trans x4 per two 32-dim blocks, on 16-bit units of 4
    // nibbles: register (cells 2t, 2t + 1; unit g) holds dims 4g .. 4g + 3
    // of the block for both cells.  Nibble e of both halves becomes the
    // fp16 pair (code - 8) exactly (OR into 1024's exponent, then minus
    // 1032; for the upper nibble of a byte 1024 + 16 code, times 1/16,
    // minus 72), and the block's scales are folded into P (fp32, then the
    // hi + lo split), as the int8 path does per 64-dim group.  Nibbles are
    // always finite and masked cells have p = 0, so no V mask is needed;
    // a masked cell's scale bits may be anything, and clamping them to
    // +-65504 keeps 0 * s == 0 (finite scales pass unchanged).
    // M-tile 2 blk + h: row g is dim 32 blk + 4g + 2h, row g + 8 the dim
    // after it.
#pragma unroll
    for (int kq = 0; kq < C::VROWB / 32; ++kq) {
      uint32_t r[4];
      ldsm_x4_t(r, st + vq[kq]);
#pragma unroll
      for (int jb = 0; jb < 2; ++jb) {
        const int blk = 2 * kq + jb;
        const int sh = 16 * (blk & 1);
        const float s0 = __half2float(__ushort_as_half((unsigned short)(sw[0][blk >> 1] >> sh)));
        const float s8 = __half2float(__ushort_as_half((unsigned short)(sw[1][blk >> 1] >> sh)));
        uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          uint32_t h01, l01, h23, l23;
          split_pair(p[nt][0] * s0, p[nt][1] * s0, h01, l01);
          split_pair(p[nt][2] * s8, p[nt][3] * s8, h23, l23);
          if constexpr (HL) {
            bh[nt][0] = movmatrix_t(t >= 2 ? l01 : h01);
            bh[nt][1] = movmatrix_t(t >= 2 ? l23 : h23);
          } else {
            bh[nt][0] = movmatrix_t(h01);
            bh[nt][1] = movmatrix_t(h23);
            bl[nt][0] = movmatrix_t(l01);
            bl[nt][1] = movmatrix_t(l23);
          }
        }
        const uint32_t wl = r[2 * jb], wh = r[2 * jb + 1];
        const uint32_t wl8 = wl >> 8, wh8 = wh >> 8;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t xl = h ? wl8 : wl, xh = h ? wh8 : wh;
          const uint32_t af[4] = {nib_lo(xl), nib_hi(xl), nib_lo(xh), nib_hi(xh)};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(o[2 * blk + h][nt], af, bh[nt][0], bh[nt][1]);
            if constexpr (!HL) mma16816(o[2 * blk + h][nt], af, bl[nt][0], bl[nt][1]);
          }
        }
      }
    }
  } else {
    const unsigned short* vsc =
        reinterpret_cast<const unsigned short*>(smem + C::SMEM_SC + s * C::SC_STAGE_B + C::KSCALE_B);
#pragma unroll
    for (int gv = 0; gv < C::NG; ++gv) {
      // p = 0 exactly for masked cells, whose scale bits may be anything
      // (even +-inf / NaN): clamping to +-65504 keeps 0 * s == 0.  Finite
      // fp16 scales pass unchanged.
      const float s0 = fmaxf(fminf(__half2float(__ushort_as_half(vsc[(cl + g) * C::NG + gv])), 65504.f), -65504.f);
      const float s8 = fmaxf(fminf(__half2float(__ushort_as_half(vsc[(cl + g + 8) * C::NG + gv])), 65504.f), -65504.f);
      uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float x0 = p[nt][0] * s0;
        const float x1 = p[nt][1] * s0;
        const float x2 = p[nt][2] * s8;
        const float x3 = p[nt][3] * s8;
        uint32_t h01, l01, h23, l23;
        split_pair(x0, x1, h01, l01);
        split_pair(x2, x3, h23, l23);
        if constexpr (HL) {
          bh[nt][0] = movmatrix_t(t >= 2 ? l01 : h01);
          bh[nt][1] = movmatrix_t(t >= 2 ? l23 : h23);
        } else {
          bh[nt][0] = movmatrix_t(h01);
          bh[nt][1] = movmatrix_t(h23);
          bl[nt][0] = movmatrix_t(l01);
          bl[nt][1] = movmatrix_t(l23);
        }
      }
      // Two ldmatrix.trans x4 per 64-dim group, on byte pairs: register
      // i of chunk c holds (cell 2t, dims 16c + 2g, +1) and (cell 2t + 1,
      // same dims) for cells +0 (i = 0) or +8 (i = 1), so m-tile c row g is
      // dim 16c + 2g and row g + 8 is dim 16c + 2g + 1.
#pragma unroll
      for (int jh = 0; jh < 2; ++jh) {
        const int c0 = gv * 4 + jh * 2;  // first 16-dim chunk of this pair
        uint32_t r[4];
        ldsm_x4_t(r, st + C::OFF_V + kstep(c0 >> 1));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t w0 = r[2 * h] ^ 0x80808080u, w8 = r[2 * h + 1] ^ 0x80808080u;
          uint32_t af[4];
          af[0] = hsub2(prmt(w0, kMagic, 0x4240u), kBias);  // dim 2g, cells 2t, 2t+1
          af[1] = hsub2(prmt(w0, kMagic, 0x4341u), kBias);  // dim 2g+1
          af[2] = hsub2(prmt(w8, kMagic, 0x4240u), kBias);  // dim 2g, cells 2t+8, 2t+9
          af[3] = hsub2(prmt(w8, kMagic, 0x4341u), kBias);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(o[c0 + h][nt], af, bh[nt][0], bh[nt][1]);
            if constexpr (!HL) mma16816(o[c0 + h][nt], af, bl[nt][0], bl[nt][1]);
          }
        }
      }
    }
  }
  };

  auto release = [&](int it) {
    // the last warp to let the stage go issues its refill
    __syncwarp();
    if (lane == 0) {
      const int s = it % C::STAGES;
      // acquire-release: this warp's reads of the stage happen before the
      // count moves, and the last warp sees every other warp's reads done
      int prev;
      asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                   : "=r"(prev)
                   : "r"(smem_u32(s_rel + s))
                   : "memory");
      if (prev == kConsumerWarps - 1) {
        s_rel[s] = 0;
        if (it + C::STAGES < n_tiles) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          int nb[MAXP];
          tile_blks(it + C::STAGES, blk_in_smem, nb);
          issue(it + C::STAGES, nb);
        }
      }
    }
  };

  // Software pipeline: q.k of tile it+1 and p.v of tile it form one
  // straight-line block, so the compiler can interleave the two; the
  // softmax of tile it+1 follows because it may rescale o.  Neither is
  // skipped for a slice without valid cells (stale or unloaded stage
  // memory): its logits are masked to -inf, so p = 0, FP16 V rows are
  // zeroed by mask and int8 V scales are clamped to finite values.
  int blk_n = slice_blk(0);
  int nv_cur = 0;
  float p_cur[NT][4];
  if (n_tiles > 0) {
    if (!mbar_wait(bar_full, 0, a.wait_limit)) {
      lost = true;
    } else {
      nv_cur = slice_nvalid(0, blk_n);
      blk_n = slice_blk(1);
      float z[NT][4];
      qk(0, z);
      softmax(nv_cur, c_begin + cl, z, p_cur);
    }
  }
  int it = 0;
  for (; it + 1 < n_tiles && !lost; ++it) {
    const int sn = (it + 1) % C::STAGES;
    if (!mbar_wait(bar_full + 8 * sn, ((it + 1) / C::STAGES) & 1, a.wait_limit)) {
      lost = true;
      break;
    }
    const int nv_next = slice_nvalid(it + 1, blk_n);
    blk_n = slice_blk(it + 2);
    float zn[NT][4];
    qk(sn, zn);
    pv(it % C::STAGES, nv_cur, p_cur);
    release(it);
    softmax(nv_next, c_begin + (it + 1) * kTC + cl, zn, p_cur);
    nv_cur = nv_next;
  }
  if (!lost && n_tiles > 0) {  // the last tile
    pv(it % C::STAGES, nv_cur, p_cur);
    release(it);
  }
  if (producer) {
    // Every copy this CTA issued has landed before the CTA can exit (waits
    // return at once in normal runs; they are bounded after a lost wait).
    const int n_all = n_tiles > n_first ? n_tiles : n_first;
    for (int it = n_all > C::STAGES ? n_all - C::STAGES : 0; it < n_all; ++it)
      (void)mbar_wait(bar_full + 8 * (it % C::STAGES), (it / C::STAGES) & 1, a.wait_limit);
  }

  // ---------------- merge the 4 warps, write the split's partial ----------------
  // Each warp's row maxima and sums go to shared memory; after one barrier
  // (every warp is past the loop, so the stages are free) each warp writes
  // its rows scaled to the CTA maximum into a slab of its own in the stage
  // memory; after a second barrier the 4 slabs are summed straight into the
  // split's partial in global memory.  A lost wait poisons the rows (NaN).
  if constexpr (HL) {
    // the hi and lo column sums of each row meet (lanes t < 2 keep them)
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[mt][0][k] += __shfl_xor_sync(kFull, o[mt][0][k], 2);
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float v = l[nt][j];
      v += __shfl_xor_sync(kFull, v, 4);
      v += __shfl_xor_sync(kFull, v, 8);
      v += __shfl_xor_sync(kFull, v, 16);
      l[nt][j] = v;
    }
  float* s_wml = reinterpret_cast<float*>(smem + C::SMEM_WML);  // [warp][RP][m, l]
  const bool wlost = __any_sync(kFull, lost);
  if (g == 0 && (!HL || t < 2)) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = row_of(nt, j);
        s_wml[(warp * RP + r) * 2 + 0] = wlost ? __int_as_float(0x7fc00000) : m[nt][j];
        s_wml[(warp * RP + r) * 2 + 1] = l[nt][j];
      }
  }
  __syncthreads();
  float* s_slab = reinterpret_cast<float*>(smem);  // [warp][R][HD] over the free stages
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = row_of(nt, j);
      if (r < Rc && (!HL || t < 2)) {
        float M = s_wml[r * 2];
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) M = fmaxf(M, s_wml[(w * RP + r) * 2]);
        const float wgt = (M == kNegInf || m[nt][j] == kNegInf) ? 0.f : fast_exp2(m[nt][j] - M);
        float* orow = s_slab + (warp * Rc + r) * HD;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          if constexpr (FMT == KVQ_F16) {  // m-tile rows g, g + 8 are dims 16 mt + g, + 8
            orow[mt * 16 + g] = wgt * o[mt][nt][j];
            orow[mt * 16 + g + 8] = wgt * o[mt][nt][2 + j];
          } else if constexpr (C::V4) {   // K8V4: dims 32 (mt / 2) + 4g + 2 (mt % 2), + 1
            *reinterpret_cast<float2*>(orow + (mt >> 1) * 32 + 4 * g + 2 * (mt & 1)) =
                make_float2(wgt * o[mt][nt][j], wgt * o[mt][nt][2 + j]);
          } else {                        // int8: dims 16 mt + 2g, + 1
            *reinterpret_cast<float2*>(orow + mt * 16 + 2 * g) =
                make_float2(wgt * o[mt][nt][j], wgt * o[mt][nt][2 + j]);
          }
        }
      }
    }
  __syncthreads();
  // this CTA's rows of the split's partial
  const size_t row0 = (((size_t)b * a.pool.n_kv + kvh) * a.nsplit + split) * a.R + r0;
  if constexpr (C::V4) {
    // K8V4: the merged rows are in the rotated basis; one warp per row sums
    // the slabs, rotates the row back (Walsh-Hadamard, divided by HD) and
    // writes it.  The combine is linear in the partials, so it needs no
    // change.
    constexpr int U = HD >= 128 ? 4 : 2, NI = HD / (32 * U);
    for (int r = warp; r < Rc; r += kConsumerWarps) {
      float x[NI][U];
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int d0 = U * lane + 32 * U * i;
#pragma unroll
        for (int e = 0; e < U; ++e) {
          const float* col = s_slab + r * HD + d0 + e;
          x[i][e] = (col[0] + col[Rc * HD]) + (col[2 * Rc * HD] + col[3 * Rc * HD]);
        }
      }
      wht_warp<U, NI>(x, lane);
      float* dst = a.ws_o + (row0 + r) * HD;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int d0 = U * lane + 32 * U * i;
        if constexpr (U == 4)
          *reinterpret_cast<float4*>(dst + d0) =
              make_float4(x[i][0] * (1.0f / HD), x[i][1] * (1.0f / HD), x[i][U > 2 ? 2 : 0] * (1.0f / HD),
                          x[i][U > 3 ? 3 : 0] * (1.0f / HD));
        else
          *reinterpret_cast<float2*>(dst + d0) = make_float2(x[i][0] * (1.0f / HD), x[i][1] * (1.0f / HD));
      }
    }
  } else
  for (int i4 = threadIdx.x; i4 < Rc * HD / 4; i4 += kThreads) {
    const float4 v0 = reinterpret_cast<const float4*>(s_slab)[i4];
    const float4 v1 = reinterpret_cast<const float4*>(s_slab + Rc * HD)[i4];
    const float4 v2 = reinterpret_cast<const float4*>(s_slab + 2 * Rc * HD)[i4];
    const float4 v3 = reinterpret_cast<const float4*>(s_slab + 3 * Rc * HD)[i4];
    reinterpret_cast<float4*>(a.ws_o + row0 * HD)[i4] =
        make_float4((v0.x + v1.x) + (v2.x + v3.x), (v0.y + v1.y) + (v2.y + v3.y),
                    (v0.z + v1.z) + (v2.z + v3.z), (v0.w + v1.w) + (v2.w + v3.w));
  }
  if (threadIdx.x < Rc) {
    const int r = threadIdx.x;
    float M = s_wml[r * 2];
    bool bad = M != M;
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) {
      const float mw = s_wml[(w * RP + r) * 2];
      bad |= mw != mw;
      M = fmaxf(M, mw);
    }
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = s_wml[(w * RP + r) * 2];
      if (M != kNegInf && mw != kNegInf) lsum = fmaf(s_wml[(w * RP + r) * 2 + 1], fast_exp2(mw - M), lsum);
    }
    *reinterpret_cast<float2*>(a.ws_ml + (row0 + r) * 2) =
        make_float2(bad ? __int_as_float(0x7fc00000) : M, lsum);
  }
}

// ---------------------------------------------------------------------------
// Final combine of the per-warp partials, launched as a programmatic
// dependent of the partial kernel: its CTAs wait on griddepcontrol until
// every partial is written.
// ---------------------------------------------------------------------------
constexpr int kCombineThreads = 256;
constexpr int kCombineBatch = 4;   // partial loads in flight per thread

template <int HD, int DV>
__global__ void __launch_bounds__(kCombineThreads, 4) combine_partials(DecodeArgs a) {
  // One CTA per (KV head, sequence, row, DV float4 columns).  Thread (js,
  // dv) merges column dv of the partials j = js, js + JS, ... online
  // (running maximum, rescaled sums; the loads of a batch issued together);
  // the JS slices then meet through warp shuffles and shared memory.  The
  // host picks DV so that one batch usually covers every partial.
  constexpr int JS = kCombineThreads / DV;
  constexpr int NW = kCombineThreads / 32;
  constexpr int CHUNKS = HD / 4 / DV;   // CTAs per row
  constexpr float kNegInf = -INFINITY;
  static_assert(DV <= 32 && HD / 4 % DV == 0, "combine shape");
  __shared__ float s_wm[NW];
  __shared__ float s_wl[NW];
  __shared__ int s_wbad[NW];
  __shared__ float4 s_wacc[NW][DV];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int r = blockIdx.z / CHUNKS, d0 = (blockIdx.z % CHUNKS) * DV * 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int dv = tid % DV, js = tid / DV;
  const int d = d0 + 4 * dv;
  // one sequence: every split slot is written (splits past the context say
  // "no cells"), so the context length need not be read
  const int nlive = a.n_seq == 1 ? a.nsplit
                                 : (int)fdiv((unsigned)(clamp_len_mma(__ldg(a.ctx_lens + b), a) +
                                                        a.split_cells - 1),
                                             a.div_split);
  const size_t base0 = ((size_t)b * a.pool.n_kv + kvh) * a.nsplit;

  float M = kNegInf, lsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  bool bad = false;
  for (int j0 = js; j0 < nlive; j0 += JS * kCombineBatch) {
    float mb[kCombineBatch], lb[kCombineBatch];
    float4 ob[kCombineBatch];
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      const int j = j0 + u * JS;
      mb[u] = kNegInf;
      lb[u] = 0.f;
      ob[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < nlive) {
        const size_t rj = (base0 + j) * a.R + r;
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.ws_ml + rj * 2));
        mb[u] = ml.x;
        lb[u] = ml.y;
        ob[u] = __ldcg(reinterpret_cast<const float4*>(a.ws_o + rj * HD + d));
      }
    }
    float bm = M;
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      bad |= mb[u] != mb[u];
      bm = fmaxf(bm, mb[u]);
    }
    if (bm == kNegInf) continue;
    const float sc = M == kNegInf ? 0.f : fast_exp2(M - bm);
    acc.x *= sc;
    acc.y *= sc;
    acc.z *= sc;
    acc.w *= sc;
    lsum *= sc;
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      if (mb[u] != kNegInf) {
        const float w = fast_exp2(mb[u] - bm);
        acc.x = fmaf(w, ob[u].x, acc.x);
        acc.y = fmaf(w, ob[u].y, acc.y);
        acc.z = fmaf(w, ob[u].z, acc.z);
        acc.w = fmaf(w, ob[u].w, acc.w);
        lsum = fmaf(w, lb[u], lsum);
      }
    }
    M = bm;
  }
  // block maximum (a warp holds 32 / DV slices; their columns share M)
  float wm = M;
#pragma unroll
  for (int off = DV; off < 32; off <<= 1) wm = fmaxf(wm, __shfl_xor_sync(kFull, wm, off));
  const bool wbad = __any_sync(kFull, bad);
  if (lane == 0) {
    s_wm[warp] = wm;
    s_wbad[warp] = wbad;
  }
  __syncthreads();
  float Mall = s_wm[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) Mall = fmaxf(Mall, s_wm[w]);
  const float sc = (M == kNegInf || Mall == kNegInf) ? 0.f : fast_exp2(M - Mall);
  acc.x *= sc;
  acc.y *= sc;
  acc.z *= sc;
  acc.w *= sc;
  lsum *= sc;
#pragma unroll
  for (int off = DV; off < 32; off <<= 1) {
    acc.x += __shfl_xor_sync(kFull, acc.x, off);
    acc.y += __shfl_xor_sync(kFull, acc.y, off);
    acc.z += __shfl_xor_sync(kFull, acc.z, off);
    acc.w += __shfl_xor_sync(kFull, acc.w, off);
    lsum += __shfl_xor_sync(kFull, lsum, off);
  }
  if (lane < DV) s_wacc[warp][lane] = acc;
  if (lane == 0) s_wl[warp] = lsum;
  __syncthreads();
  if (tid < DV) {
    float4 sum = s_wacc[0][tid];
    float lam = s_wl[0];
    int any_bad = s_wbad[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
      const float4 v = s_wacc[w][tid];
      sum.x += v.x;
      sum.y += v.y;
      sum.z += v.z;
      sum.w += v.w;
      lam += s_wl[w];
      any_bad |= s_wbad[w];
    }
    // an empty context (no live partial) gives 0; a lost wait gives NaN
    const float inv = lam > 0.f ? 1.f / lam : 0.f;
    float4 res = make_float4(sum.x * inv, sum.y * inv, sum.z * inv, sum.w * inv);
    if (any_bad) {
      const float nan = __int_as_float(0x7fc00000);
      res = make_float4(nan, nan, nan, nan);
    }
    const int w = div_g(a, r), gg = r - w * a.G;
    *reinterpret_cast<float4*>(a.out + (((size_t)b * a.W + w) * a.n_q + (size_t)kvh * a.G + gg) * HD +
                               d0 + 4 * tid) = res;
  }
}

template <int HD, int DV>
cudaError_t launch_combine_dv(const DecodeArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cc = {};
  cc.gridDim = dim3(a.pool.n_kv, a.n_seq, a.R * (HD / 4 / DV));
  cc.blockDim = dim3(kCombineThreads);
  cc.stream = s;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cc.attrs = pdl;
  cc.numAttrs = 1;
  return cudaLaunchKernelEx(&cc, combine_partials<HD, DV>, a);
}

// Widest column block (fewest CTAs) whose slices still cover every partial
// slot in one batch of loads; 4 columns (64 slices) when none does.
template <int HD>
cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s) {
  const int need_js = (a.nsplit + kCombineBatch - 1) / kCombineBatch;
  constexpr int MAXDV = HD / 4 < 32 ? HD / 4 : 32;
  if (need_js <= kCombineThreads / 32 && MAXDV >= 32) return launch_combine_dv<HD, MAXDV>(a, s);
  if (need_js <= kCombineThreads / 16 && MAXDV >= 16) return launch_combine_dv<HD, 16>(a, s);
  if (need_js <= kCombineThreads / 8) return launch_combine_dv<HD, 8>(a, s);
  return launch_combine_dv<HD, 4>(a, s);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
}

// Span sp of one codes array: [total rows][span bytes] starting at byte
// sp * span of each row (rows of row_bytes), box = one piece of cells, the
// swizzle as wide as the span (32, 64 or 128 bytes).
bool make_map(CUtensorMap* map, const void* base, int span, int row_bytes, int sp, long long rows,
              int piece_cells) {
  auto enc = encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)span, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)span, (cuuint32_t)piece_cells};
  const cuuint32_t estr[2] = {1, 1};
  void* span_base = static_cast<char*>(const_cast<void*>(base)) + (size_t)sp * span;
  const CUtensorMapSwizzle sw = span == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : span == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, span_base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Resident CTAs per SM of one configuration (0 if it cannot run), after
// raising its dynamic shared-memory limit; done once per context.
template <int FMT, int HD, int NT, bool HL>
int ctas_per_sm_impl() {
  static ContextCache<int> cache;
  int occ = 0;
  const bool ok = per_context(cache, &occ, [](int* v) {
    using C = Cfg<FMT, HD, NT>;
    if (cudaFuncSetAttribute(decode_mma<FMT, HD, NT, HL>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return false;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma<FMT, HD, NT, HL>, kThreads,
                                                      C::SMEM) != cudaSuccess)
      return false;
    *v = n;
    return true;
  });
  return ok ? occ : 0;
}

template <int FMT, int HD, int NT, bool HL>
cudaError_t launch_impl(const DecodePlan& p, const DecodeArgs& a, cudaStream_t s) {
  using C = Cfg<FMT, HD, NT>;
  if (ctas_per_sm_impl<FMT, HD, NT, HL>() <= 0) return cudaErrorInvalidConfiguration;
  const long long rows = (long long)a.pool.n_blocks * a.pool.n_kv << a.pool.bs_log2;
  const int piece = 1 << (a.pool.bs_log2 < 6 ? a.pool.bs_log2 : 6);
  TmaMaps maps;
  memset(&maps, 0, sizeof(maps));
  for (int sp = 0; sp < C::NCH; ++sp)
    if (!make_map(&maps.k[sp], a.pool.k, C::SWB, C::ROWB, sp, rows, piece)) return cudaErrorInvalidValue;
  for (int sp = 0; sp < C::VNCH; ++sp)
    if (!make_map(&maps.v[sp], a.pool.v, C::VSWB, C::VROWB, sp, rows, piece)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  const long long items = (long long)p.nsplit * a.pool.n_kv * a.n_seq * a.n_rt;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  cfg.gridDim = dim3((unsigned)items);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_mma<FMT, HD, NT, HL>, maps, a);
  if (e != cudaSuccess) return e;
  return launch_combine<HD>(a, s);
}

// Kernel shape of a row count: 0 = one 8-column tile with hi/lo columns
// (at most 4 rows), else the number of 8-row tiles.
int tile_code(int rows) { return rows <= 4 ? 0 : rows <= 8 ? 1 : rows <= 16 ? 2 : rows <= 32 ? 4 : -1; }

template <int FMT, int HD>
int ctas_per_sm_hd(int code) {
  switch (code) {
    case 0: return ctas_per_sm_impl<FMT, HD, 1, true>();
    case 1: return ctas_per_sm_impl<FMT, HD, 1, false>();
    case 2: if constexpr (HD <= 128) return ctas_per_sm_impl<FMT, HD, 2, false>(); break;
    case 4: if constexpr (HD <= 64) return ctas_per_sm_impl<FMT, HD, 4, false>(); break;
  }
  return 0;
}

template <int FMT, int HD>
cudaError_t launch_hd(int code, const DecodePlan& p, const DecodeArgs& a, cudaStream_t s) {
  switch (code) {
    case 0: return launch_impl<FMT, HD, 1, true>(p, a, s);
    case 1: return launch_impl<FMT, HD, 1, false>(p, a, s);
    case 2: if constexpr (HD <= 128) return launch_impl<FMT, HD, 2, false>(p, a, s); break;
    case 4: if constexpr (HD <= 64) return launch_impl<FMT, HD, 4, false>(p, a, s); break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace

void* tensor_map_encoder() {
  static void* fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = f;
  });
  return fn;
}

unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
    (void)cudaGetLastError();
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

bool mma_decode_supported(int fmt, int hd, int rows) {
  if (rows < 1 || rows > 32) return false;
  if (hd != 64 && hd != 128 && hd != 256) return false;
  return fmt == KVQ_F16 || fmt == KVQ_Q8 || fmt == KVQ_K8V4;
}

// Query rows one CTA holds: 8-row MMA tiles while their fp32 accumulators
// (HD / 16 m-tiles x 4 floats per tile and thread) stay at 32 per thread
// or fewer -- 32 rows at head_dim 64, 16 at 128, 8 at 256.
int mma_rows_per_cta(int hd) { return 8 * (256 / hd); }

int mma_cell_tile() { return kTC; }

int mma_ctas_per_sm(int fmt, int hd, int rows) {
  const int nt = tile_code(rows);
  if (fmt == KVQ_F16) {
    if (hd == 64) return ctas_per_sm_hd<KVQ_F16, 64>(nt);
    if (hd == 128) return ctas_per_sm_hd<KVQ_F16, 128>(nt);
    return ctas_per_sm_hd<KVQ_F16, 256>(nt);
  }
  if (fmt == KVQ_Q8) {
    if (hd == 64) return ctas_per_sm_hd<KVQ_Q8, 64>(nt);
    if (hd == 128) return ctas_per_sm_hd<KVQ_Q8, 128>(nt);
    return ctas_per_sm_hd<KVQ_Q8, 256>(nt);
  }
  if (hd == 64) return ctas_per_sm_hd<KVQ_K8V4, 64>(nt);
  if (hd == 128) return ctas_per_sm_hd<KVQ_K8V4, 128>(nt);
  return ctas_per_sm_hd<KVQ_K8V4, 256>(nt);
}

cudaError_t launch_decode_mma_partial(int fmt, int hd, const DecodePlan& p, const DecodeArgs& a,
                                      cudaStream_t s) {
  const int nt = tile_code(p.rt_rows);
  if (fmt == KVQ_F16) {
    if (hd == 64) return launch_hd<KVQ_F16, 64>(nt, p, a, s);
    if (hd == 128) return launch_hd<KVQ_F16, 128>(nt, p, a, s);
    return launch_hd<KVQ_F16, 256>(nt, p, a, s);
  }
  if (fmt == KVQ_Q8) {
    if (hd == 64) return launch_hd<KVQ_Q8, 64>(nt, p, a, s);
    if (hd == 128) return launch_hd<KVQ_Q8, 128>(nt, p, a, s);
    return launch_hd<KVQ_Q8, 256>(nt, p, a, s);
  }
  if (hd == 64) return launch_hd<KVQ_K8V4, 64>(nt, p, a, s);
  if (hd == 128) return launch_hd<KVQ_K8V4, 128>(nt, p, a, s);
  return launch_hd<KVQ_K8V4, 256>(nt, p, a, s);
}

}  // namespace kvq

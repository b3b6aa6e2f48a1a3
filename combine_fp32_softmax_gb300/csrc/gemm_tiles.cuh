#pragma once
// Tile machinery shared by the persistent grouped GEMM kernels and the
// forward MegaKernel: grouped GEMM over ragged expert segments on tcgen05
// tensor cores.
//
// The expert FFN of the MoE layer runs as GroupGEMM -> SwiGLU -> GroupGEMM
// (UniEP page, "Unified Expert-Parallel MoE MegaKernel for LLM Training",
// section 1.1), padding-free over segments of different lengths with
// per-segment pointer arithmetic (same page, section 2.2, scoreboard
// paragraph).  The backward's weight gradients are the transposed GroupGEMM
// whose reduction runs over each expert's tokens (section 1.1); each such sum
// runs in ascending row order inside one CTA so the bits never depend on the
// schedule.  The persistent, one-CTA-per-SM design follows the persistent
// worker model of section 2.2 and the streaming-GEMM argument of the
// AutoOverlap page, section 2.1 (no per-expert launches, no partial waves).
//
// Design (one CTA per SM, 192 threads; CG = 1 or 2 CTAs per tile):
//   warp 0      TMA producer: 128B-swizzled tiles of A (128 x 64) and B
//               (256 x 64, or this CTA's 128 x 64 half on a CTA pair) into
//               a shared-memory ring: 4 stages of 48 KB (one CTA per
//               tile), 6 of 32 KB (pairs).  MN-major operands come as one
//               3D box per operand (map3d_mn).
//   warp 1      allocates 512 TMEM columns, issues tcgen05.mma from one lane
//               (M=128, or M=256 on a pair from the even CTA; N=256, K=16,
//               bf16 -> fp32), commits to mbarriers (multicast to both
//               CTAs of a pair); a ragged-K tail's last partial 16-row step
//               is zeroed in shared memory.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (one TMEM lane per
//               thread = one output row), fused elementwise work, results
//               staged through swizzled shared memory and written with TMA
//               tensor stores (coalesced, asynchronous).  Warps whose 32
//               rows are not all valid (a segment's last m-tile) store
//               their valid rows directly.  The dH epilogue TMA-loads its
//               elementwise inputs ([a|b]) per warp, double-buffered,
//               and stages its outputs in the buffer the inputs came in.
//               The weight-gradient kinds run warps 2-9: two per TMEM lane
//               quadrant, each on half of the tile's columns.  The fp32
//               kinds can instead store straight from registers
//               (epilogue_f32_direct, a runtime option).
//   The accumulator is double-buffered in TMEM (2 x 256 columns) so the
//   epilogue of tile i overlaps the main loop of tile i+1.
// Tiles of equal length are taken in a static round-robin over CTAs, those of
// the weight-gradient kinds from a ticket counter (grouped_gemm.cu); either
// way every output element is produced by exactly one tile with a fixed K
// order.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "ptx.cuh"
#include "trace.h"

namespace moe {
namespace {

constexpr int kMaxStages = 7;
// Tile numbers in flight from the ticket-taking producer to the other roles
// (dynamic tile scheduling of the grouped GEMM kernels).
constexpr int kTileRing = 8;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBBytes = kBN * kBK * 2;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 48 KB (one CTA per tile)
constexpr int kBoxBytes = 64 * 64 * 2;          // one MN-major box: 64 x 64 bf16
constexpr int kMaxSeg = 256 + 4;
constexpr int kEpiWarps = 4;                  // epilogue warps of most kinds (one per TMEM lane quadrant)
constexpr int kMaxEpiWarps = 8;               // the weight-gradient kinds: two per quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;
// Position of the calling warp among the epilogue warps (warps 2, 3, ...).
__device__ __forceinline__ int epi_warp() { return static_cast<int>(threadIdx.x >> 5) - 2; }
constexpr int kTmemCols = 512;
constexpr int kChunkBytes = 32 * 64;  // one staged chunk: 32 rows x 64 bytes (SW64)

struct GemmParams {
  CUtensorMap tmA0, tmA1, tmB0, tmB1;  // operands
  CUtensorMap tmO0, tmO1;              // outputs written with TMA stores
  CUtensorMap tmX0;                    // dH epilogue input: [a|b]
  int T, d, f, E, k, S, R;
  int N;       // output columns per expert
  int Mw;      // ragged-K kinds: output rows per expert
  int K;       // ragged-M kinds: reduction length
  int nt_dh;   // dH: column tiles per row (number of partial dot products)
  int has_ab;  // GEMM 1: save [a|b]
  int prefetch_kb;  // K blocks of a CTA's next tile brought into L2 ahead of its loads
  int tile_order;   // ragged-K kinds: 0 = longest segments first, 1 = long segments' tiles interleaved
  int nst;          // pipeline stages in use (at most Pipe<KIND, CG>::STAGES)
  int epi_direct;   // fp32-output kinds: 1 = epilogue stores straight from registers (no staging)
  const int32_t* offsets;
  const int32_t* row_slot;
  const float* topk_w;
  void* out0;
  void* out1;
  float* out_partial;
  int* err;
};

template <int KIND>
struct Traits {
  static constexpr bool A_MN = (KIND == kDW13 || KIND == kDW2);
  static constexpr bool B_MN = (KIND == kDH || KIND == kDX || KIND == kDW13 || KIND == kDW2);
  static constexpr bool RAGGED_K = (KIND == kDW13 || KIND == kDW2);
  static constexpr int BNE = (KIND == kG1) ? 128 : 256;  // output columns per tile

  static constexpr int STAGES = 4;
  // fp32 kinds: 16-column chunks, two staging buffers in flight.
  static constexpr int F32_ROUNDS = 2;
  // per epilogue warp: GEMM 1 one chunk of Hw, a, b; dH two buffers of two
  // chunks, each taking a chunk's [a, b] inputs and then, in place, its
  // dA, dB outputs; fp32 kinds F32_ROUNDS output chunks.
  static constexpr int EPI_BYTES = (KIND == kG1)   ? 3 * kChunkBytes
                                   : (KIND == kDH) ? 4 * kChunkBytes
                                                   : F32_ROUNDS * kChunkBytes;
};

// Shared-memory pipeline of one kind.  CG = 1: one CTA per 128 x 256 tile,
// 48 KB stages.  CG = 2: a CTA pair per 256 x 256 tile (tcgen05 CTA group of
// two): each CTA stages its 128 rows of A and its half of B's 256 columns,
// 32 KB a stage, so more stages fit and B is fetched once per 256 rows.
template <int KIND, int CG>
struct Pipe {
  static constexpr int TILE_M = kBM * CG;  // output rows per (pair) tile
  static constexpr int B_BYTES = kBBytes / CG;
  static constexpr int B_BOXES = 4 / CG;  // MN-major B: 64-column boxes per CTA
  static constexpr int STAGE_BYTES = kABytes + B_BYTES;
  // Epilogue warps of the stand-alone kernel: two per TMEM lane quadrant,
  // each taking half of a tile's columns, for the weight-gradient kinds
  // (their short-K tiles finish the MMAs about as fast as four warps move
  // 256 fp32 columns out).  dH keeps four: one warp sums a row's dw dot over
  // the whole tile, and eight would cost it a pipeline stage.
  static constexpr int EPI_WARPS = (KIND == kDW13 || KIND == kDW2) ? kMaxEpiWarps : kEpiWarps;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int STAGES = CG == 1 ? Traits<KIND>::STAGES : 6;
};

struct SharedState {
  uint64_t full[kMaxStages], empty[kMaxStages], tfull[2], tempty[2], drain;
  uint64_t ready[kMaxStages];  // CG = 2, even CTA: the odd CTA's stage has landed
  // dH epilogue input buffers, two per epilogue warp (indexed by the warp's
  // position among the epilogue warps, never by its TMEM lane quadrant: two
  // warps share a quadrant when a kind runs eight)
  uint64_t aux[kMaxEpiWarps][2];
  uint64_t tile_full[kTileRing], tile_empty[kTileRing];  // tile-number ring
  int tile_ring[kTileRing];
  uint32_t tmem_base;
  int abort;
  int nseg;
  int total_tiles;
  int tiles_per_seg;  // ragged-K kinds: every segment has the same tile count
  int long_tiles;     // ragged-K kinds, interleaved order: tiles of the long segments (0: plain order)
  int long_span;      // ... spread evenly over the first long_span tickets
  int seg_row0[kMaxSeg];
  union {
    int prefix[kMaxSeg + 1];  // ragged-M kinds: tiles before each segment
    int order[kMaxSeg];       // ragged-K kinds: segments by descending rows
  };
};

// Rows of segment s: routed expert s owns [offsets[s], offsets[s+1]); the
// shared experts own T rows each.
__device__ __forceinline__ int seg_rows(const GemmParams& p, const SharedState& ss, int s) {
  if (s >= p.E) return p.T;
  return (s + 1 < p.E ? ss.seg_row0[s + 1] : p.R) - ss.seg_row0[s];
}

// Shared memory one CTA can have (the sm_100 family's per-block opt-in).
constexpr int kSmemBudget = 232448;

// Shared memory of the stand-alone kernel: the ring, the epilogue staging
// (none when the fp32 kinds store straight from registers) and the state.
template <int KIND, int CG = 1>
constexpr int smem_bytes(bool direct = false) {
  return Pipe<KIND, CG>::STAGES * Pipe<KIND, CG>::STAGE_BYTES +
         (direct ? 0 : Pipe<KIND, CG>::EPI_WARPS * Traits<KIND>::EPI_BYTES) + static_cast<int>(sizeof(SharedState));
}
// Pipeline stages with direct epilogue stores: the staging memory they do
// not need takes more of the ring (CTA pairs: a seventh 32 KB stage).
template <int KIND, int CG = 1>
constexpr int direct_stages() {
  constexpr bool fp32_out = KIND == kG2 || KIND == kDX || KIND == kDW13 || KIND == kDW2;
  constexpr int fit = (kSmemBudget - static_cast<int>(sizeof(SharedState))) / Pipe<KIND, CG>::STAGE_BYTES;
  return !fp32_out ? Pipe<KIND, CG>::STAGES : (fit < kMaxStages ? fit : kMaxStages);
}
template <int KIND, int CG = 1>
constexpr int direct_smem_bytes() {
  return direct_stages<KIND, CG>() * Pipe<KIND, CG>::STAGE_BYTES + static_cast<int>(sizeof(SharedState));
}
// The larger of the two modes' footprints (what a launch asks for).
template <int KIND, int CG = 1>
constexpr int launch_smem_bytes() {
  return smem_bytes<KIND, CG>() > direct_smem_bytes<KIND, CG>() ? smem_bytes<KIND, CG>()
                                                                 : direct_smem_bytes<KIND, CG>();
}

// One CTA's part of a tile.  m0 and rows are this CTA's: in a pair the odd
// CTA's part starts 128 rows further and may hold no valid row (`active`
// false: it still takes part in the main loop, and writes nothing).
struct TileInfo {
  int seg, m0, n0, rows, grow0, nkb;
  bool shared, active;
};

// Bounded wait that ignores the abort flag (used to drain in-flight copies).
__device__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

template <int KIND, int CG>
__device__ __forceinline__ int tiles_of(const GemmParams& p, int rows) {
  using Tr = Traits<KIND>;
  constexpr int TM = Pipe<KIND, CG>::TILE_M;
  const int ntn = (p.N + Tr::BNE - 1) / Tr::BNE;
  if constexpr (Tr::RAGGED_K)
    return ((p.Mw + TM - 1) / TM) * ntn;
  else
    return ((rows + TM - 1) / TM) * ntn;
}

// Segment table: routed expert e owns GEMM rows [offsets[e], offsets[e+1]);
// shared expert s owns [R + s*T, R + (s+1)*T).  prefix[] counts tiles.
template <int KIND, int CG = 1>
__device__ void build_segments(const GemmParams& p, SharedState& ss) {
  const int nseg = p.E + p.S;
  for (int s = threadIdx.x; s < nseg; s += blockDim.x)
    ss.seg_row0[s] = (s < p.E) ? p.offsets[s] : p.R + (s - p.E) * p.T;
  __syncthreads();
  if (kDebug && threadIdx.x == 0) {  // the routing tables' segment starts: 0, non-decreasing, ending at R
    bool ok = ss.seg_row0[0] == 0 && p.offsets[p.E] == p.R;
    for (int s = 1; s < p.E; ++s) ok = ok && ss.seg_row0[s] >= ss.seg_row0[s - 1];
    debug_ok(ok, p.err, kDbgSegments + KIND, blockIdx.x);
  }
  if constexpr (Traits<KIND>::RAGGED_K) {
    // Longest segments first: their tiles (K = their rows) are spread over
    // the CTAs before the short ones fill in, so no long tile ends the
    // launch alone.  Stable rank: more rows first, then lower index.
    for (int s = threadIdx.x; s < nseg; s += blockDim.x) {
      const int n = seg_rows(p, ss, s);
      int rank = 0;
      for (int u = 0; u < nseg; ++u) {
        const int m = seg_rows(p, ss, u);
        rank += (m > n || (m == n && u < s)) ? 1 : 0;
      }
      ss.order[rank] = s;
    }
    if (threadIdx.x == 0) {
      ss.tiles_per_seg = tiles_of<KIND, CG>(p, 0);
      ss.total_tiles = ss.tiles_per_seg * nseg;
      ss.nseg = nseg;
      // Interleaved order: a segment is long if it has more than twice the
      // mean rows of the non-empty segments.  The long segments (first in
      // `order`) are compute-heavy per output byte, the short ones
      // write-heavy; spreading the long ones' tiles over the first 3/4 of
      // the tickets keeps both kinds running side by side, and the last
      // long tile still starts early enough to end with the rest.
      ss.long_tiles = 0;
      ss.long_span = 0;
      if (p.tile_order == 1) {
        long long total_rows = 0;
        int nonempty = 0;
        for (int u = 0; u < nseg; ++u) {
          const int m = seg_rows(p, ss, u);
          total_rows += m;
          nonempty += m > 0 ? 1 : 0;
        }
        int nlong = 0;
        while (nlong < nseg && static_cast<long long>(seg_rows(p, ss, ss.order[nlong])) * nonempty > 2 * total_rows)
          ++nlong;
        if (nlong > 0 && nlong < nseg) {
          ss.long_tiles = nlong * ss.tiles_per_seg;
          ss.long_span = max(ss.long_tiles, static_cast<int>((3ll * ss.total_tiles) / 4));
        }
      }
    }
  } else if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (nseg + 31) / 32;
    const int lo = min(nseg, lane * per), hi = min(nseg, lo + per);
    int local = 0;
    for (int s = lo; s < hi; ++s) local += tiles_of<KIND, CG>(p, seg_rows(p, ss, s));
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    int run = incl - local;
    for (int s = lo; s < hi; ++s) {
      ss.prefix[s] = run;
      run += tiles_of<KIND, CG>(p, seg_rows(p, ss, s));
    }
    if (lane == 31) {
      ss.prefix[nseg] = incl;
      ss.total_tiles = incl;
      ss.nseg = nseg;
    }
  }
  __syncthreads();
}

template <int KIND, int CG = 1>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, const SharedState& ss, int tile,
                                                int rank = 0) {
  using Tr = Traits<KIND>;
  int lo = 0, hi = ss.nseg;
  int pos = tile;  // ragged-K kinds: position in the segment order (segment-major)
  if constexpr (Tr::RAGGED_K) {  // equal tile counts per segment, taken in ss.order
    if (ss.long_tiles > 0) {
      // Long tile j sits at ticket floor(j * span / NL); the count of long
      // positions <= i is ceil((i + 1) * NL / span), capped at NL.  Short
      // tiles fill the other tickets in order.
      const long long NL = ss.long_tiles, span = ss.long_span;
      auto nlong_upto = [&](long long i) { return i < 0 ? 0ll : min(NL, ((i + 1) * NL + span - 1) / span); };
      const long long c = nlong_upto(tile), cprev = nlong_upto(tile - 1);
      pos = static_cast<int>(c > cprev ? c - 1 : NL + (tile - c));
    }
    lo = ss.order[pos / ss.tiles_per_seg];
  } else {
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ss.prefix[mid] <= tile)
        lo = mid;
      else
        hi = mid;
    }
  }
  TileInfo t;
  t.seg = lo;
  t.shared = lo >= p.E;
  const int local = Tr::RAGGED_K ? pos % ss.tiles_per_seg : tile - ss.prefix[lo];
  const int ntn = (p.N + Tr::BNE - 1) / Tr::BNE;
  const int mb = local / ntn, nb = local - mb * ntn;
  t.m0 = mb * Pipe<KIND, CG>::TILE_M + rank * kBM;
  t.n0 = nb * Tr::BNE;
  if constexpr (Tr::RAGGED_K) {
    t.rows = seg_rows(p, ss, lo);
    t.grow0 = ss.seg_row0[lo];
    t.nkb = (t.rows + kBK - 1) / kBK;
    t.active = t.m0 < p.Mw;
  } else {
    t.rows = min(kBM, seg_rows(p, ss, lo) - t.m0);
    t.grow0 = ss.seg_row0[lo] + t.m0;
    t.nkb = p.K / kBK;
    t.active = t.rows > 0;
  }
  if constexpr (kDebug) {  // the tile's rows lie inside the GEMM rows (TMA boxes start inside their tensor)
    const long long rs = static_cast<long long>(p.R) + static_cast<long long>(p.S) * p.T;
    const bool ok = t.grow0 >= 0 && (!t.active || static_cast<long long>(t.grow0) + t.rows <= rs);
    if (!debug_ok(ok, p.err, kDbgTmaCoord + KIND, tile)) t.active = false;
  }
  return t;
}

// Ragged-K kinds: the last K block of a tile whose segment length is not a
// multiple of 16 (the MMA's K step).  Its rows from the segment end up to the
// next multiple of 16 are zeroed in shared memory; K steps wholly past the
// end are not issued.
template <int KIND>
__device__ __forceinline__ bool is_k_tail(const TileInfo& t, int kb) {
  return Traits<KIND>::RAGGED_K && kb == t.nkb - 1 && (t.rows & 15) != 0;
}
// K steps (16 rows each) of block kb that hold rows of the segment.
template <int KIND>
__device__ __forceinline__ int k_steps(const TileInfo& t, int kb) {
  if constexpr (Traits<KIND>::RAGGED_K)
    return min(kBK / 16, (t.rows - kb * kBK + 15) >> 4);
  else
    return kBK / 16;
}

// The last column tile of dH and dW2 when it holds at most 128 of the f
// columns (f = 1408 leaves 128 of 256): its MMAs are N = 128 and its B boxes
// half as wide, instead of spending half of each 256-wide MMA on zeros.  A
// pair then splits B 64 + 64 columns.
template <int KIND>
__device__ __forceinline__ bool narrow_tile(const GemmParams& p, const TileInfo& t) {
  if constexpr (KIND == kDH || KIND == kDW2)
    return p.N - t.n0 <= kBN / 2;
  else
    return false;
}

// One stage of TMA loads: A (this CTA's 128 rows) and this CTA's part of B
// (all 256 columns for CG = 1; columns [128 rank, 128 rank + 128) for
// CG = 2).  Boxes that fall outside a tensor are zero-filled.  `to_even`:
// completion is counted on the pair's even CTA's barrier.
// PREFETCH: the same boxes are only brought into L2.
template <int KIND, int CG = 1, bool PREFETCH = false>
__device__ __forceinline__ void issue_loads(const GemmParams& p, const TileInfo& t, int kb, uint8_t* sA,
                                            uint8_t* sB, uint64_t* bar, int rank = 0, bool to_even = false) {
  auto tma_load_2d = [&](void* dst, const CUtensorMap* map, uint64_t* b, int c0, int c1) {
    if constexpr (PREFETCH)
      tma_prefetch_2d(map, c0, c1);
    else if (CG == 2 && to_even)
      tma_load_2d_to_even(dst, map, b, c0, c1);
    else
      moe::tma_load_2d(dst, map, b, c0, c1);
  };
  // MN-major operand: rows [row, row + 64) and columns [col, col + 64 n) in one
  // instruction (a 3D box of n 64-column chunks, see map3d_mn); the single
  // producer lane issues every load, so fewer instructions keep it ahead.
  auto tma_load_mn = [&](void* dst, const CUtensorMap* map, uint64_t* b, int col, int row) {
    if constexpr (PREFETCH)
      tma_prefetch_3d(map, 0, row, col / 64);
    else if (CG == 2 && to_even)
      tma_load_3d_to_even(dst, map, b, 0, row, col / 64);
    else
      moe::tma_load_3d(dst, map, b, 0, row, col / 64);
  };
  const int kk = kb * kBK;
  const bool narrow = narrow_tile<KIND>(p, t);
  const int bn0 = t.n0 + (narrow ? 64 : 128) * rank;  // first B column this CTA stages
  const CUtensorMap* mapB = narrow ? &p.tmB1 : &p.tmB0;  // dH, dW2: tmB1 holds half the 64-column chunks
  if constexpr (KIND == kG1) {
    // accumulator columns [0,128) = gate rows of W1, [128,256) = up rows of W3
    tma_load_2d(sA, t.shared ? &p.tmA1 : &p.tmA0, bar, kk, t.shared ? t.m0 : t.grow0);
    if (CG == 1 || rank == 0) tma_load_2d(sB, &p.tmB0, bar, kk, t.seg * p.f + t.n0);
    if (CG == 1 || rank == 1) tma_load_2d(sB + (CG == 1 ? kBBytes / 2 : 0), &p.tmB1, bar, kk, t.seg * p.f + t.n0);
  } else if constexpr (KIND == kG2) {
    tma_load_2d(sA, &p.tmA0, bar, kk, t.grow0);
    tma_load_2d(sB, &p.tmB0, bar, kk, t.seg * p.d + bn0);
  } else if constexpr (KIND == kDH) {
    tma_load_2d(sA, t.shared ? &p.tmA1 : &p.tmA0, bar, kk, t.shared ? t.m0 : t.grow0);
    tma_load_mn(sB, mapB, bar, bn0, t.seg * p.d + kk);
  } else if constexpr (KIND == kDX) {
    tma_load_2d(sA, &p.tmA0, bar, kk, t.grow0);
    const bool second = kk >= p.f;
    const int krow = t.seg * p.f + (second ? kk - p.f : kk);
    tma_load_mn(sB, second ? &p.tmB1 : &p.tmB0, bar, bn0, krow);
  } else if constexpr (KIND == kDW13) {
    tma_load_mn(sA, &p.tmA0, bar, t.m0, t.grow0 + kk);
    tma_load_mn(sB, t.shared ? &p.tmB1 : &p.tmB0, bar, bn0, t.shared ? kk : t.grow0 + kk);
  } else {  // kDW2
    tma_load_mn(sA, t.shared ? &p.tmA1 : &p.tmA0, bar, t.m0, t.shared ? kk : t.grow0 + kk);
    tma_load_mn(sB, mapB, bar, bn0, t.grow0 + kk);
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void tmem_ld_32x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 16 TMEM lanes x 4 repetitions of 256 bits (8 consecutive 32-bit columns
// each): thread t of the warp gets, for repetition j, lane (base + t/4)
// columns 8j + 2(t%4) + {0, 1} in r[4j], r[4j+1] and lane (base + 8 + t/4)
// the same columns in r[4j+2], r[4j+3].
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// One row of a 32-row x 64-byte staging chunk in the TMA 64-byte swizzle
// layout: 16-byte piece c of row r sits at piece c ^ ((r >> 1) & 3).  A
// warp writing or reading one row per lane touches every bank once per
// eight lanes (no bank conflicts).
__device__ __forceinline__ void stage_row64(uint8_t* buf, int row, const uint32_t* w) {
  const int sw = (row >> 1) & 3;
  uint4* r = reinterpret_cast<uint4*>(buf + row * 64);
#pragma unroll
  for (int c = 0; c < 4; ++c) r[c ^ sw] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}
__device__ __forceinline__ void load_row64(const uint8_t* buf, int row, uint32_t* w) {
  const int sw = (row >> 1) & 3;
  const uint4* r = reinterpret_cast<const uint4*>(buf + row * 64);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = r[c ^ sw];
    w[4 * c] = v.x;
    w[4 * c + 1] = v.y;
    w[4 * c + 2] = v.z;
    w[4 * c + 3] = v.w;
  }
}
// Direct (unstaged) store of 16 words: the fallback for rows of warps that
// are only partly inside the segment.
__device__ __forceinline__ void store_words16(void* dst, const uint32_t* w) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < 4; ++c) d[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

// Per-epilogue-warp state carried across tiles.
struct EpiState {
  int it = 0;             // tiles done (TMEM buffer / phase)
  uint32_t chunks = 0;    // staged chunks issued in the current tile
  uint32_t auxn = 0;      // dH input chunks loaded so far (buffer = auxn & 1)
  uint32_t auxpar = 0;    // next wait parity of each dH input buffer
  uint32_t auxpend = 0;   // dH input buffers with a load in flight
  float w = 1.f;          // GEMM 2, dH: this lane's row's routing weight, read before the accumulator is ready
};

// The routing weight of the lane's row (1 for shared rows and rows past the
// segment), read while the tile's main loop still runs.
__device__ __forceinline__ float row_weight(const GemmParams& p, const TileInfo& t, int q) {
  const int r = 32 * q + (threadIdx.x & 31);
  if (!(r < t.rows && !t.shared)) return 1.f;
  const int slot = p.row_slot[static_cast<size_t>(t.grow0) + r];
  if (!debug_ok(static_cast<unsigned>(slot) < static_cast<unsigned>(p.R), p.err, kDbgEpiRow, t.grow0 + r)) return 0.f;
  return p.topk_w[slot];
}

// Staging helper: lane 0 waits until earlier chunks stopped reading the
// buffer about to be rewritten.
template <int MAX_PENDING>
__device__ __forceinline__ void staging_reuse_wait(uint32_t chunks) {
  if (chunks > MAX_PENDING) {
    if ((threadIdx.x & 31) == 0) bulk_wait_read<MAX_PENDING>();
    __syncwarp();
  }
}
__device__ __forceinline__ void staging_publish() {
  fence_proxy_async_smem();
  __syncwarp();
}

// fp32 outputs (GEMM 2, dX, dW1/dW3, dW2): 16-column chunks, double-buffered.
template <int KIND>
__device__ __forceinline__ void epilogue_f32(const GemmParams& p, const TileInfo& t, int q, uint32_t tacc,
                                             uint8_t* stg, EpiState& es, int part = 0, int nparts = 1) {
  const int lane = threadIdx.x & 31;
  const int r = 32 * q + lane;  // tile row of this lane
  const CUtensorMap* map = &p.tmO0;
  int orow0;                    // tensor-map row of the warp's first row
  float* optr;                  // this lane's output row (fallback path)
  bool full, rowok;
  int N;
  if constexpr (KIND == kG2 || KIND == kDX) {
    N = p.d;
    rowok = r < t.rows;
    full = t.rows >= 32 * q + 32;
    const size_t grow = static_cast<size_t>(t.grow0) + r;
    orow0 = t.grow0 + 32 * q;
    optr = static_cast<float*>(p.out0) + grow * N;
  } else if constexpr (KIND == kDW13) {
    N = p.d;
    const int mw0 = t.m0 + 32 * q;  // the warp's 32 rows all sit in dW1 or all in dW3 (f % 32 == 0)
    const bool second = mw0 >= p.f;
    map = second ? &p.tmO1 : &p.tmO0;
    orow0 = t.seg * p.f + (second ? mw0 - p.f : mw0);
    optr = static_cast<float*>(second ? p.out1 : p.out0) + (static_cast<size_t>(orow0) + lane) * N;
    rowok = full = true;
  } else {  // kDW2
    N = p.f;
    const int m = t.m0 + r;
    rowok = m < p.d;
    full = t.m0 + 32 * q + 32 <= p.d;
    orow0 = t.seg * p.d + t.m0 + 32 * q;
    optr = static_cast<float*>(p.out0) + (static_cast<size_t>(t.seg) * p.d + m) * N;
  }
  const bool zero = Traits<KIND>::RAGGED_K && t.nkb == 0;  // empty expert: exact zeros
  constexpr int NR = Traits<KIND>::F32_ROUNDS;
  // this warp's chunks: [j0, j1) of the tile's 16-column chunks
  const int per = 16 / nparts;
  const int j0 = part * per, j1 = min(min(16, (N - t.n0 + 15) / 16), j0 + per);
  es.chunks = 0;
  if (j0 >= j1) return;
  // Software pipeline: chunk j+1's TMEM load is in flight while chunk j is
  // staged and its TMA store issued.
  uint32_t cur[16], nxt[16];
  if (zero) {
#pragma unroll
    for (int i = 0; i < 16; ++i) cur[i] = 0u;
  } else {
    tmem_ld_32x16(tacc + 16 * j0, cur);
    tmem_ld_wait();
  }
#pragma unroll 1
  for (int j = j0; j < j1; ++j) {
    const bool more = j + 1 < j1;
    if (more && !zero) tmem_ld_32x16(tacc + 16 * (j + 1), nxt);
    const int n = t.n0 + 16 * j;
    if (full) {
      uint8_t* buf = stg + (es.chunks % NR) * kChunkBytes;
      staging_reuse_wait<NR - 1>(es.chunks);
      stage_row64(buf, lane, cur);
      staging_publish();
      if (lane == 0) {
        tma_store_2d(map, buf, n, orow0);
        bulk_commit();
      }
      ++es.chunks;
    } else if (rowok) {
      store_words16(optr + n, cur);
    }
    if (more) {
      if (!zero) tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) cur[i] = zero ? 0u : nxt[i];
    }
  }
}

// fp32 outputs written straight from registers (no shared-memory staging).
// Each group of 32 accumulator columns is read as two 16-lane halves in the
// 16x256b shape, and one exchange between neighbouring threads leaves every
// thread 4 consecutive columns of one row: a warp store then covers 8 rows x
// 64 contiguous bytes (two full 32-byte sectors per row).  Rows and columns
// outside the output are not written; the same values as epilogue_f32.
template <int KIND>
__device__ __forceinline__ void epilogue_f32_direct(const GemmParams& p, const TileInfo& t, int q, uint32_t tacc,
                                                    EpiState& es, int part = 0, int nparts = 1) {
  const int lane = threadIdx.x & 31;
  const int quad = lane >> 2, c = lane & 3;
  int N;
  float* base;       // output element (row 32q of this warp, column 0)
  long long ld;      // row stride in elements
  int valid_rows;    // rows of this warp (from 32q) that exist
  if constexpr (KIND == kG2 || KIND == kDX) {
    N = p.d;
    ld = N;
    base = static_cast<float*>(p.out0) + (static_cast<size_t>(t.grow0) + 32 * q) * N;
    valid_rows = t.rows - 32 * q;
  } else if constexpr (KIND == kDW13) {
    N = p.d;
    ld = N;
    const int mw0 = t.m0 + 32 * q;
    const bool second = mw0 >= p.f;
    base = static_cast<float*>(second ? p.out1 : p.out0) +
           (static_cast<size_t>(t.seg) * p.f + (second ? mw0 - p.f : mw0)) * N;
    valid_rows = 32;
  } else {  // kDW2
    N = p.f;
    ld = N;
    base = static_cast<float*>(p.out0) + (static_cast<size_t>(t.seg) * p.d + t.m0 + 32 * q) * N;
    valid_rows = p.d - t.m0 - 32 * q;
  }
  const bool zero = Traits<KIND>::RAGGED_K && t.nkb == 0;  // empty expert: exact zeros
  // this warp's columns: [g0, ncols) of the tile, in groups of 32
  const int span = 256 / nparts;
  const int g0 = part * span;
  const int ncols = min(min(256, N - t.n0), g0 + span);
  es.chunks = 0;
  if (g0 >= ncols) return;
  // Software pipeline: group g+1's two TMEM loads are in flight while group
  // g is exchanged and stored.
  uint32_t v[2][16], nv[2][16];
  if (zero) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[0][i] = v[1][i] = 0u;
  } else {
    tmem_ld_16x256b_x4(tacc + g0, v[0]);
    tmem_ld_16x256b_x4(tacc + (16u << 16) + g0, v[1]);
    tmem_ld_wait();
  }
#pragma unroll 1
  for (int g = g0; g < ncols; g += 32) {
    const bool more = g + 32 < ncols;
    if (more && !zero) {
      tmem_ld_16x256b_x4(tacc + g + 32, nv[0]);
      tmem_ld_16x256b_x4(tacc + (16u << 16) + g + 32, nv[1]);
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {       // rows quad (sub 0) and quad + 8 (sub 1) of this half
        const int row = 16 * half + 8 * sub + quad;
#pragma unroll
        for (int jp = 0; jp < 2; ++jp) {        // repetitions 2jp and 2jp + 1
          const int j0 = 2 * jp, j1 = 2 * jp + 1;
          const uint32_t* a = &v[half][4 * j0 + 2 * sub];
          const uint32_t* b = &v[half][4 * j1 + 2 * sub];
          // even threads keep repetition j0 and take the odd neighbour's j0;
          // odd threads keep j1 and take the even neighbour's j1
          const bool odd = c & 1;
          const uint32_t s0 = __shfl_xor_sync(0xffffffffu, odd ? a[0] : b[0], 1);
          const uint32_t s1 = __shfl_xor_sync(0xffffffffu, odd ? a[1] : b[1], 1);
          float4 o;
          int col;
          if (!odd) {
            o = make_float4(__uint_as_float(a[0]), __uint_as_float(a[1]), __uint_as_float(s0), __uint_as_float(s1));
            col = g + 8 * j0 + 2 * c;
          } else {
            o = make_float4(__uint_as_float(s0), __uint_as_float(s1), __uint_as_float(b[0]), __uint_as_float(b[1]));
            col = g + 8 * j1 + 2 * (c - 1);
          }
          if (row < valid_rows && t.n0 + col < N)
            *reinterpret_cast<float4*>(base + static_cast<long long>(row) * ld + t.n0 + col) = o;
        }
      }
    }
    if (more) {
      if (!zero) tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        v[0][i] = zero ? 0u : nv[0][i];
        v[1][i] = zero ? 0u : nv[1][i];
      }
    }
  }
}

// GEMM 1: columns [0,128) of the accumulator hold a (gate), [128,256) hold b
// (up) for outputs n0..n0+127; Hw = bf16(w * (silu(a) * b)) with the row's
// routing weight (1 for shared rows), optionally [a|b].
__device__ __forceinline__ void epilogue_g1(const GemmParams& p, const TileInfo& t, int q, uint32_t tacc,
                                            uint8_t* stg, EpiState& es) {
  const int lane = threadIdx.x & 31;
  const int r = 32 * q + lane;
  const bool rowok = r < t.rows, full = t.rows >= 32 * q + 32;
  const size_t grow = static_cast<size_t>(t.grow0) + r;
  const int orow0 = t.grow0 + 32 * q;
  uint16_t* Hw = static_cast<uint16_t*>(p.out0);
  uint16_t* AB = static_cast<uint16_t*>(p.out1);
  const float w = es.w;
  es.chunks = 0;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    const int n = t.n0 + 32 * c;
    if (n >= p.f) break;
    uint32_t a[32], b[32];
    tmem_ld_32x32(tacc + 32 * c, a);
    tmem_ld_32x32(tacc + 128 + 32 * c, b);
    tmem_ld_wait();
    uint32_t hp[16], ap[16], bp[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float a0 = __uint_as_float(a[2 * i]), a1 = __uint_as_float(a[2 * i + 1]);
      const float b0 = __uint_as_float(b[2 * i]), b1 = __uint_as_float(b[2 * i + 1]);
      hp[i] = pack_bf16(w * (__fdividef(a0, 1.f + __expf(-a0)) * b0), w * (__fdividef(a1, 1.f + __expf(-a1)) * b1));
      ap[i] = pack_bf16(a0, a1);
      bp[i] = pack_bf16(b0, b1);
    }
    if (full) {
      staging_reuse_wait<0>(es.chunks);
      stage_row64(stg, lane, hp);
      if (p.has_ab) {
        stage_row64(stg + kChunkBytes, lane, ap);
        stage_row64(stg + 2 * kChunkBytes, lane, bp);
      }
      staging_publish();
      if (lane == 0) {
        tma_store_2d(&p.tmO0, stg, n, orow0);
        if (p.has_ab) {
          tma_store_2d(&p.tmO1, stg + kChunkBytes, n, orow0);
          tma_store_2d(&p.tmO1, stg + 2 * kChunkBytes, p.f + n, orow0);
        }
        bulk_commit();
      }
      ++es.chunks;
    } else if (rowok) {
      store_words16(Hw + grow * p.f + n, hp);
      if (p.has_ab) {
        store_words16(AB + grow * 2 * p.f + n, ap);
        store_words16(AB + grow * 2 * p.f + p.f + n, bp);
      }
    }
  }
}

// dH: inputs a, b of the tile's 32-column chunks are TMA-loaded per warp
// into two buffers (2 chunks of 2 KB each); a chunk's outputs dA, dB are
// staged in the buffer its inputs came in, which is refilled (two chunks
// ahead) once the output stores have read it.  Sharing the buffers this way
// leaves room for six pipeline stages on CTA pairs.  h for the dw dot is
// formed again from the same bf16 a and b (the forward kept only w * h), so
// dH reads 2 and writes 2 bf16 values per element.
__device__ __forceinline__ int dh_chunks(const GemmParams& p, const TileInfo& t) {
  return min(8, (p.f - t.n0 + 31) / 32);
}
// This warp's chunks [c0, c1): all of them, or half with two warps per quadrant.
__device__ __forceinline__ int2 dh_range(const GemmParams& p, const TileInfo& t, int part, int nparts) {
  const int nch = dh_chunks(p, t), per = 8 / nparts;
  return make_int2(min(nch, part * per), min(nch, (part + 1) * per));
}
__device__ __forceinline__ void dh_issue_inputs(const GemmParams& p, const TileInfo& t, int q, int c, uint8_t* stg,
                                                SharedState& ss, EpiState& es) {
  const int buf = es.auxn & 1;
  ++es.auxn;
  if ((threadIdx.x & 31) == 0) {
    uint8_t* in = stg + buf * 2 * kChunkBytes;
    uint64_t* bar = &ss.aux[epi_warp()][buf];
    const int n = t.n0 + 32 * c, row0 = t.grow0 + 32 * q;
    mbar_arrive_expect_tx(bar, 2 * kChunkBytes);
    tma_load_2d(in, &p.tmX0, bar, n, row0);                    // a
    tma_load_2d(in + kChunkBytes, &p.tmX0, bar, p.f + n, row0);  // b
  }
  es.auxpend |= 1u << buf;
}
// Issued before the tile's accumulator is ready so the loads overlap the wait.
__device__ __forceinline__ void dh_prefetch(const GemmParams& p, const TileInfo& t, int q, uint8_t* stg,
                                            SharedState& ss, EpiState& es, int part, int nparts) {
  const int2 r = dh_range(p, t, part, nparts);
  if (r.x < r.y) dh_issue_inputs(p, t, q, r.x, stg, ss, es);
  if (r.x + 1 < r.y) dh_issue_inputs(p, t, q, r.x + 1, stg, ss, es);
}

// The dw partial dot of a row is summed over the tile's 256 columns in chunk
// order by the one warp that covers the row, and stored at index n0 / 256.
__device__ __forceinline__ bool epilogue_dh(const GemmParams& p, const TileInfo& t, int q, uint32_t tacc,
                                            uint8_t* stg, SharedState& ss, EpiState& es, volatile int* abort,
                                            int where, int part, int nparts) {
  const int lane = threadIdx.x & 31;
  const int r = 32 * q + lane;
  const bool rowok = r < t.rows, full = t.rows >= 32 * q + 32;
  const size_t grow = static_cast<size_t>(t.grow0) + r;
  const int orow0 = t.grow0 + 32 * q;
  const float w = es.w;
  uint16_t* dAB = static_cast<uint16_t*>(p.out0);
  const int2 range = dh_range(p, t, part, nparts);
  const int c0 = range.x, c1 = range.y;
  const uint32_t first = es.auxn - min(2, c1 - c0);  // input chunk index of chunk c0
  float dot = 0.f;
  es.chunks = 0;
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    const int n = t.n0 + 32 * c;
    const int buf = (first + (c - c0)) & 1;
    if (!mbar_wait(&ss.aux[epi_warp()][buf], (es.auxpar >> buf) & 1, abort, p.err, where)) return false;
    es.auxpar ^= 1u << buf;
    es.auxpend &= ~(1u << buf);
    uint32_t g[32];
    tmem_ld_32x32(tacc + 32 * c, g);
    tmem_ld_wait();
    const uint8_t* in = stg + buf * 2 * kChunkBytes;
    uint32_t aw[16], bw[16];
    load_row64(in, lane, aw);
    load_row64(in + kChunkBytes, lane, bw);
    // every lane has its rows in registers: the buffer now takes the outputs
    __syncwarp();
    uint32_t ra[16], rb[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      float dA2[2], dB2[2];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float a = half ? bf16_hi(aw[u]) : bf16_lo(aw[u]);
        const float b = half ? bf16_hi(bw[u]) : bf16_lo(bw[u]);
        const float graw = __uint_as_float(g[2 * u + half]);
        const float s = __fdividef(1.f, 1.f + __expf(-a));
        const float as = a * s;
        dot += graw * (as * b);
        const float dH = w * graw;
        dA2[half] = dH * b * s * (1.f + a * (1.f - s));
        dB2[half] = dH * as;
      }
      ra[u] = pack_bf16(dA2[0], dA2[1]);
      rb[u] = pack_bf16(dB2[0], dB2[1]);
    }
    uint8_t* out = stg + buf * 2 * kChunkBytes;
    if (full) {
      // Each lane overwrites only the row it read.
      stage_row64(out, lane, ra);
      stage_row64(out + kChunkBytes, lane, rb);
      staging_publish();
      if (lane == 0) {
        tma_store_2d(&p.tmO0, out, n, orow0);
        tma_store_2d(&p.tmO0, out + kChunkBytes, p.f + n, orow0);
        bulk_commit();
        if (c + 2 < c1) bulk_wait_read<0>();  // the stores have read the buffer before it is refilled
      }
      __syncwarp();
      ++es.chunks;
    } else {
      if (rowok) {
        store_words16(dAB + grow * 2 * p.f + n, ra);
        store_words16(dAB + grow * 2 * p.f + p.f + n, rb);
      }
      fence_proxy_async_smem();  // the inputs' generic reads before the refill's TMA writes
      __syncwarp();
    }
    if (c + 2 < c1) dh_issue_inputs(p, t, q, c + 2, stg, ss, es);
  }
  if (rowok && !t.shared) p.out_partial[grow * p.nt_dh + t.n0 / kBN] = dot;
  return true;
}

// ---------------------------------------------------------- per-tile roles
// Shared by the grouped GEMM kernels and the MegaKernel, so a tile's MMA
// sequence and epilogue arithmetic are the same code in both.

// CG = 2: the even CTA's tempty barriers count the epilogue warps of both
// CTAs; ready[s] takes the odd CTA's word that its part of stage s landed.
// tile_empty (used in the even CTA, or the only one) counts every role that
// reads a tile number from the ring: the MMA warp and the epilogue warps of
// both CTAs, and the odd CTA's producer.
template <int CG = 1, int EW = kEpiWarps>
__device__ __forceinline__ void init_gemm_barriers(SharedState& ss) {
  for (int i = 0; i < kTileRing; ++i) {
    mbar_init(&ss.tile_full[i], 1);
    mbar_init(&ss.tile_empty[i], CG == 2 ? 2 * (1 + EW) + 1 : 1 + EW);
  }
  for (int s = 0; s < kMaxStages; ++s) {
    mbar_init(&ss.full[s], 1);
    mbar_init(&ss.empty[s], 1);
    mbar_init(&ss.ready[s], 1);
  }
  for (int a = 0; a < 2; ++a) {
    mbar_init(&ss.tfull[a], 1);
    mbar_init(&ss.tempty[a], EW * CG);
  }
  for (int w = 0; w < EW; ++w) {
    mbar_init(&ss.aux[w][0], 1);
    mbar_init(&ss.aux[w][1], 1);
  }
  mbar_init(&ss.drain, 1);
  ss.abort = 0;
}

// Producer lane: every K block of one tile through the NST-stage ring.
// filled / fill_par: stages with a load counted on this CTA's own barrier,
// and the parity of the phase it completes (for the drain on abort).
struct ProducerState {
  int stage = 0;
  uint32_t phase = 0, filled = 0, fill_par = 0;
  uint32_t tail_par = 0;  // CG = 2, odd CTA: phase parity of its own full[s] (turns on K tails only)
};

// CG = 2: both CTAs' loads of a stage are counted on the even CTA's full[s]
// (the even CTA expects both CTAs' bytes), so no thread stands between the
// odd CTA's data and the MMA.  A ragged-K tail is the exception: each CTA's
// loads complete on its own full[s], each zeroes its own rows past the
// segment end, and the odd CTA then arrives on the even CTA's ready[s].
template <int KIND, int CG = 1>
__device__ __forceinline__ bool produce_tile(const GemmParams& p, const TileInfo& t, SharedState& ss, uint8_t* smem,
                                             ProducerState& ps, volatile int* abort, int where, int NST, int rank = 0) {
  constexpr int SB = Pipe<KIND, CG>::STAGE_BYTES;
  // bytes one CTA's loads of a stage bring (half of B on a narrow tile)
  const int sb = narrow_tile<KIND>(p, t) ? SB - Pipe<KIND, CG>::B_BYTES / 2 : SB;
  for (int kb = 0; kb < t.nkb; ++kb) {
    if (!mbar_wait(&ss.empty[ps.stage], ps.phase ^ 1, abort, p.err, where)) return false;
    uint8_t* sA = smem + ps.stage * SB;
    const uint32_t bit = 1u << ps.stage;
    const bool tail = CG == 2 && is_k_tail<KIND>(t, kb);
    if (CG == 1 || rank == 0 || tail) mbar_arrive_expect_tx(&ss.full[ps.stage], CG == 2 && !tail ? 2 * sb : sb);
    issue_loads<KIND, CG>(p, t, kb, sA, sA + kABytes, &ss.full[ps.stage], rank, CG == 2 && rank == 1 && !tail);
    if (CG == 1 || rank == 0) {
      ps.filled |= bit;
      ps.fill_par = (ps.fill_par & ~bit) | (ps.phase << ps.stage);
    } else if (tail) {
      ps.filled |= bit;
      ps.fill_par = (ps.fill_par & ~bit) | (ps.tail_par & bit);
      ps.tail_par ^= bit;
    }
    if (++ps.stage == NST) {
      ps.stage = 0;
      ps.phase ^= 1;
    }
  }
  return true;
}

// The first K blocks of a tile this CTA will load next, into L2: the loads
// of the current tile then overlap the DRAM latency of the next one (short-K
// tiles of a new segment otherwise all start with misses).
template <int KIND, int CG = 1>
__device__ __forceinline__ void prefetch_tile(const GemmParams& p, const TileInfo& t, int rank = 0) {
  const int n = min(t.nkb, p.prefetch_kb);
  for (int kb = 0; kb < n; ++kb) issue_loads<KIND, CG, true>(p, t, kb, nullptr, nullptr, nullptr, rank);
}

// Lets every copy the producer issued land before the CTA may exit.
__device__ __forceinline__ void producer_drain(SharedState& ss, const ProducerState& ps) {
  for (int s = 0; s < kMaxStages; ++s)
    if (ps.filled & (1u << s)) mbar_wait_drain(&ss.full[s], (ps.fill_par >> s) & 1);
}

// MMA warp: one tile into TMEM accumulator buffer `it & 1`; lane 0 issues.
struct MmaState {
  int stage = 0, it = 0;
  uint32_t phase = 0;
  uint32_t tail_par = 0;  // CG = 2: parity of ready[s] (even CTA) / own full[s] (odd CTA) on K tails
  bool issued = false;
};

// Ragged-K tail: in the last K step that holds rows of the segment, the
// rows past the segment's end (they hold the next segment's rows) are
// zeroed in shared memory, in every box of A and B, so they add nothing.
// Both operands are zeroed so that a non-finite value of another expert's
// rows cannot reach this expert's sums.  MN-major boxes hold one K row per
// 128 bytes; all 8 pieces of a row are cleared, so the swizzle is moot.
template <int KIND, int CG>
__device__ __forceinline__ void zero_k_tail(const TileInfo& t, int kb, uint8_t* sA, uint8_t* sB) {
  if (!is_k_tail<KIND>(t, kb)) return;
  const int kvalid = t.rows - kb * kBK;
  const int n = (((kvalid + 15) & ~15) - kvalid) * 8;  // 16-byte pieces per box, < 128
  const int lane = threadIdx.x & 31;
  constexpr int NBOX = 2 + Pipe<KIND, CG>::B_BOXES;
#pragma unroll
  for (int box = 0; box < NBOX; ++box) {
    uint8_t* bb = (box < 2) ? sA + box * kBoxBytes : sB + (box - 2) * kBoxBytes;
    for (int idx = lane; idx < n; idx += 32)
      reinterpret_cast<uint4*>(bb + (kvalid + (idx >> 3)) * 128)[idx & 7] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// MMA warp, one tile.  CG = 1, or the even CTA of a pair: waits for the
// accumulator buffer, then per stage for its data (on a pair's ragged-K
// tail also for the odd CTA's word that its zeroed part is ready), issues
// the MMAs from lane 0 and commits: stage release to the producers (both
// CTAs of a pair), and the finished accumulator to the epilogues (both
// CTAs).  The odd CTA's MMA warp only handles ragged-K tails: waits for its
// own stage, zeroes its rows past the segment end and tells the even CTA.
template <int KIND, int CG = 1>
__device__ __forceinline__ bool mma_tile(const GemmParams& p, const TileInfo& t, SharedState& ss, uint8_t* smem,
                                         uint32_t tmem, MmaState& ms, volatile int* abort, int where, int NST,
                                         int rank = 0) {
  using Tr = Traits<KIND>;
  constexpr int SB = Pipe<KIND, CG>::STAGE_BYTES;
  constexpr uint32_t kIdescFull = idesc_bf16_f32(kBM * CG, kBN, Tr::A_MN ? 1 : 0, Tr::B_MN ? 1 : 0);
  constexpr uint32_t kIdescNarrow = idesc_bf16_f32(kBM * CG, kBN / 2, Tr::A_MN ? 1 : 0, Tr::B_MN ? 1 : 0);
  const uint32_t kIdesc = narrow_tile<KIND>(p, t) ? kIdescNarrow : kIdescFull;
  const int lane = threadIdx.x & 31;
  if (CG == 2 && rank == 1) {
    // The odd CTA's MMA warp only zeroes its part of ragged-K tails, but it
    // walks every tile's K blocks, so its ring position stays that of the
    // pair when a launch mixes kinds.
    for (int kb = 0; kb < t.nkb; ++kb) {
      if constexpr (Tr::RAGGED_K) {
        if (is_k_tail<KIND>(t, kb)) {
          const uint32_t bit = 1u << ms.stage;
          if (!mbar_wait(&ss.full[ms.stage], (ms.tail_par & bit) ? 1u : 0u, abort, p.err, where | (1 << 20)))
            return false;
          ms.tail_par ^= bit;
          uint8_t* sA = smem + ms.stage * SB;
          zero_k_tail<KIND, CG>(t, kb, sA, sA + kABytes);
          if (lane == 0) mbar_arrive_rank(&ss.ready[ms.stage], 0);
          __syncwarp();
        }
      }
      if (++ms.stage == NST) {
        ms.stage = 0;
        ms.phase ^= 1;
      }
    }
    return true;
  }
  const int acc = ms.it & 1;
  const uint32_t aph = (ms.it >> 1) & 1;
  ++ms.it;
  if (!mbar_wait<CG == 2>(&ss.tempty[acc], aph ^ 1, abort, p.err, where)) return false;
  tc_fence_after();
  const uint32_t dtm = tmem + acc * kBN;
  for (int kb = 0; kb < t.nkb; ++kb) {
    if (!mbar_wait(&ss.full[ms.stage], ms.phase, abort, p.err, where | (1 << 20))) return false;
    uint8_t* sA = smem + ms.stage * SB;
    uint8_t* sB = sA + kABytes;
    if constexpr (Tr::RAGGED_K) zero_k_tail<KIND, CG>(t, kb, sA, sB);
    if constexpr (CG == 2 && Tr::RAGGED_K) {
      if (is_k_tail<KIND>(t, kb)) {
        const uint32_t bit = 1u << ms.stage;
        if (!mbar_wait<true>(&ss.ready[ms.stage], (ms.tail_par & bit) ? 1u : 0u, abort, p.err,
                             where | (3 << 20)))
          return false;
        ms.tail_par ^= bit;
      }
    }
    tc_fence_after();
    if (lane == 0) {
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      const int nk4 = k_steps<KIND>(t, kb);
#pragma unroll
      for (int k4 = 0; k4 < kBK / 16; ++k4) {
        if (k4 >= nk4) break;
        const uint64_t ad = Tr::A_MN ? smem_desc_sw128(a0 + k4 * 2048, kBoxBytes, 1024)
                                     : smem_desc_sw128(a0 + k4 * 32, 16, 1024);
        const uint64_t bd = Tr::B_MN ? smem_desc_sw128(b0 + k4 * 2048, kBoxBytes, 1024)
                                     : smem_desc_sw128(b0 + k4 * 32, 16, 1024);
        umma_bf16<CG>(dtm, ad, bd, kIdesc, (kb | k4) != 0 ? 1u : 0u);
      }
      if constexpr (CG == 2)
        umma_commit_pair(&ss.empty[ms.stage]);
      else
        umma_commit(&ss.empty[ms.stage]);
      ms.issued = true;
    }
    __syncwarp();
    if (++ms.stage == NST) {
      ms.stage = 0;
      ms.phase ^= 1;
    }
  }
  if (lane == 0) {
    if constexpr (CG == 2)
      umma_commit_pair(&ss.tfull[acc]);
    else
      umma_commit(&ss.tfull[acc]);
  }
  __syncwarp();
  return true;
}

// Waits for the tensor core before TMEM is released on an aborted run.
template <int CG = 1>
__device__ __forceinline__ void mma_drain(SharedState& ss, const MmaState& ms) {
  if ((threadIdx.x & 31) == 0 && ms.issued) {
    umma_commit<CG>(&ss.drain);
    mbar_wait_drain(&ss.drain, 0);
  }
  __syncwarp();
}

// Epilogue warp (2..5): one tile out of TMEM buffer `es.it & 1`.  `stg` is
// this warp's staging memory.  The TMEM buffer is released as soon as the
// last accumulator load is done; the staged stores drain in the background
// and are waited for (read side) before the staging memory is reused.
// In a pair the odd CTA's warps release the buffer on the even CTA's
// barrier.  A part with no valid row still waits for the accumulator, so its
// release cannot count toward an earlier phase of the barrier.
template <int KIND, int CG = 1, int EW = kEpiWarps>
__device__ __forceinline__ bool epilogue_step(const GemmParams& p, const TileInfo& t, SharedState& ss, uint32_t tmem,
                                              uint8_t* stg, EpiState& es, volatile int* abort, int where,
                                              int rank = 0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lanes [32q, 32q+32) are reachable from this warp
  // with two warps per TMEM lane quadrant, each takes half of the columns
  constexpr int NP = EW / kEpiWarps;
  const int part = NP > 1 ? (warp - 2) / kEpiWarps : 0;
  static_assert(KIND != kDH || NP == 1, "one warp sums a row's dw partial dot over the whole tile");
  const int acc = es.it & 1;
  const uint32_t aph = (es.it >> 1) & 1;
  ++es.it;
  if constexpr (KIND == kDH)
    if (t.active) dh_prefetch(p, t, q, stg, ss, es, part, NP);
  if constexpr (KIND == kG1 || KIND == kDH)
    if (t.active) es.w = row_weight(p, t, q);
  if (!mbar_wait(&ss.tfull[acc], aph, abort, p.err, where)) return false;
  tc_fence_after();
  const uint32_t tacc = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN;
  bool ok = true;
  if (!t.active) {
  } else if constexpr (KIND == kG1)
    epilogue_g1(p, t, q, tacc, stg, es);
  else if constexpr (KIND == kDH)
    ok = epilogue_dh(p, t, q, tacc, stg, ss, es, abort, where, part, NP);
  else
  {
    if (p.epi_direct)
      epilogue_f32_direct<KIND>(p, t, q, tacc, es, part, NP);
    else
      epilogue_f32<KIND>(p, t, q, tacc, stg, es, part, NP);
  }
  tc_fence_before();
  __syncwarp();
  if (ok && lane == 0) {
    if (CG == 2 && rank == 1)
      mbar_arrive_rank(&ss.tempty[acc], 0);
    else
      mbar_arrive(&ss.tempty[acc]);
  }
  if (lane == 0) bulk_wait_read<0>();  // staging memory free for the next tile
  __syncwarp();
  return ok;
}

// Before an epilogue warp may leave: its TMA stores complete and its
// in-flight input loads landed.
__device__ __forceinline__ void epilogue_drain(SharedState& ss, const EpiState& es) {
  if ((threadIdx.x & 31) == 0) {
    bulk_wait_all();
    for (int b = 0; b < 2; ++b)
      if (es.auxpend & (1u << b)) mbar_wait_drain(&ss.aux[epi_warp()][b], (es.auxpar >> b) & 1);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ host
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Row-major matrix [outer, inner] of bf16 (esize 2) or fp32 (esize 4) seen
// as 2D boxes of box_outer rows x box_inner elements; out-of-range reads
// fill zeros and out-of-range parts of a stored box are skipped.
bool map2d_any(CUtensorMap* m, const void* base, int esize, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !base || inner == 0 || outer == 0) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * esize};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// Operand tiles: bf16, 64-element (128-byte) swizzled rows.
bool map2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  return map2d_any(m, base, 2, inner, outer, box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}
// MN-major operand tiles: a row-major bf16 matrix [rows, cols] (cols a
// multiple of 64) seen as 3D {64 columns of a chunk, row, chunk} (strides
// cols*2 and 128 bytes).  A box {64, 64 rows, chunks} lands in shared memory
// as `chunks` consecutive 64 x 64 blocks of 8 KB with 128-byte swizzled rows:
// the layout the MN-major UMMA descriptor reads (8 KB between 64-element
// groups), fetched by one instruction instead of one per block.
bool map3d_mn(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t chunks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !base || cols == 0 || rows == 0 || cols % 64) return false;
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {cols * 2, 128};
  const cuuint32_t box[3] = {64, 64, chunks};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// Epilogue chunks: 32 rows x 64 bytes (32 bf16 or 16 fp32), 64-byte swizzle.
bool map_chunk_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer) {
  return map2d_any(m, base, 2, inner, outer, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}
bool map_chunk_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer) {
  return map2d_any(m, base, 4, inner, outer, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Tensor maps and pointers of one GEMM kind (CG: CTAs per tile).
template <int KIND, int CG = 1>
bool fill_params(const GemmArgs& a, GemmParams& p) {
  std::memset(&p, 0, sizeof(p));
  const uint64_t T = a.T, d = a.d, f = a.f, nexp = a.E + a.S, R = uint64_t(a.T) * a.k, Rs = R + uint64_t(a.S) * a.T;
  p.T = a.T;
  p.d = a.d;
  p.f = a.f;
  p.E = a.E;
  p.k = a.k;
  p.S = a.S;
  p.R = static_cast<int>(R);
  p.offsets = a.offsets;
  p.row_slot = a.row_slot;
  p.topk_w = a.topk_w;
  p.err = a.err;
  p.nt_dh = ceil_div(a.f, kBN);
  bool ok = true;
  auto alt = [](const void* want, const void* fallback) { return want ? want : fallback; };
  if constexpr (KIND == kG1) {
    ok &= map2d(&p.tmA0, a.Xp, d, R, 64, 128);
    ok &= map2d(&p.tmA1, alt(a.x, a.Xp), d, a.x ? T : R, 64, 128);
    ok &= map2d(&p.tmB0, a.W1, d, nexp * f, 64, 128);
    ok &= map2d(&p.tmB1, a.W3, d, nexp * f, 64, 128);
    ok &= map_chunk_bf16(&p.tmO0, a.Hw_out, f, Rs);
    p.has_ab = a.AB_out != nullptr;
    if (p.has_ab) ok &= map_chunk_bf16(&p.tmO1, a.AB_out, 2 * f, Rs);
    p.N = a.f;
    p.K = a.d;
    p.out0 = a.Hw_out;
    p.out1 = a.AB_out;
  } else if constexpr (KIND == kG2) {
    ok &= map2d(&p.tmA0, a.Hw, f, Rs, 64, 128);
    ok &= map2d(&p.tmB0, a.W2, f, nexp * d, 64, 256 / CG);
    ok &= map_chunk_f32(&p.tmO0, a.Op_out, d, Rs);
    p.N = a.d;
    p.K = a.f;
    p.out0 = a.Op_out;
  } else if constexpr (KIND == kDH) {
    ok &= map2d(&p.tmA0, a.G, d, R, 64, 128);
    ok &= map2d(&p.tmA1, a.dy, d, T, 64, 128);
    ok &= map3d_mn(&p.tmB0, a.W2, f, nexp * d, 4 / CG);
    ok &= map3d_mn(&p.tmB1, a.W2, f, nexp * d, 2 / CG);  // narrow last column tile
    ok &= map_chunk_bf16(&p.tmO0, a.dAB_out, 2 * f, Rs);
    ok &= map_chunk_bf16(&p.tmX0, a.AB, 2 * f, Rs);
    p.N = a.f;
    p.K = a.d;
    p.out0 = a.dAB_out;
    p.out_partial = a.partial_out;
  } else if constexpr (KIND == kDX) {
    ok &= map2d(&p.tmA0, a.dAB, 2 * f, Rs, 64, 128);
    ok &= map3d_mn(&p.tmB0, a.W1, d, nexp * f, 4 / CG);
    ok &= map3d_mn(&p.tmB1, a.W3, d, nexp * f, 4 / CG);
    ok &= map_chunk_f32(&p.tmO0, a.dXp_out, d, Rs);
    p.N = a.d;
    p.K = 2 * a.f;
    p.out0 = a.dXp_out;
  } else if constexpr (KIND == kDW13) {
    ok &= map3d_mn(&p.tmA0, a.dAB, 2 * f, Rs, 2);
    ok &= map3d_mn(&p.tmB0, a.Xp, d, R, 4 / CG);
    ok &= map3d_mn(&p.tmB1, alt(a.x, a.Xp), d, a.x ? T : R, 4 / CG);
    ok &= map_chunk_f32(&p.tmO0, a.dW1_out, d, nexp * f);
    ok &= map_chunk_f32(&p.tmO1, a.dW3_out, d, nexp * f);
    p.Mw = 2 * a.f;
    p.N = a.d;
    p.out0 = a.dW1_out;
    p.out1 = a.dW3_out;
  } else {
    ok &= map3d_mn(&p.tmA0, a.G, d, R, 2);
    ok &= map3d_mn(&p.tmA1, a.dy, d, T, 2);
    ok &= map3d_mn(&p.tmB0, a.Hw, f, Rs, 4 / CG);
    ok &= map3d_mn(&p.tmB1, a.Hw, f, Rs, 2 / CG);  // narrow last column tile
    ok &= map_chunk_f32(&p.tmO0, a.dW2_out, f, nexp * d);
    p.Mw = a.d;
    p.N = a.f;
    p.out0 = a.dW2_out;
  }
  return ok;
}

}  // namespace
}  // namespace moe

// Persistent grouped GEMM over ragged expert segments on tcgen05 tensor cores
// (one kernel per GEMM kind; the tile machinery is in gemm_tiles.cuh).
//
// Warp roles, shared-memory ring, TMEM double buffering and the staged TMA
// epilogues are described in gemm_tiles.cuh.  Tiles of equal length (the
// ragged-M kinds) are taken in a static round-robin over the CTAs.  Tiles of
// the ragged-K kinds (weight gradients: K = the segment's rows, so a shared
// expert's tiles are many times longer than a routed expert's) are handed
// out dynamically: the producer of each CTA (the even CTA of each pair)
// takes tile numbers from a launch-wide ticket counter, longest segments
// first, and passes them to the CTA's other roles (and the odd CTA's)
// through a small ring in shared memory; a CTA that drew long tiles simply
// takes fewer short ones.  Which CTA computes a tile does not matter to the
// result: every output element is produced by exactly one tile with a fixed
// K order.
#include <algorithm>
#include <cstring>

#include "gemm_tiles.cuh"

namespace moe {
namespace {

// Even CTA (or the only one): publishes the tile number of the i-th ticket
// (-1: no more tiles) to its ring and, for a pair, to the odd CTA's, once
// every role has read the slot's previous number.
template <int CG>
__device__ __forceinline__ bool feed_put(SharedState& ss, int i, int tile, volatile int* abort, int* err,
                                         int where) {
  const int slot = i % kTileRing;
  const uint32_t par = (i / kTileRing) & 1;
  if (!mbar_wait<CG == 2>(&ss.tile_empty[slot], par ^ 1, abort, err, where)) return false;
  ss.tile_ring[slot] = tile;
  if constexpr (CG == 2) {
    st_shared_rank(&ss.tile_ring[slot], 1, tile);
    mbar_arrive_rank(&ss.tile_full[slot], 1);  // release at cluster scope: the store above is seen first
  }
  mbar_arrive(&ss.tile_full[slot]);
  return true;
}

// Every role but the ticket taker: the i-th tile number (-1: none left, or
// the launch is aborting).  All lanes of the calling warp read it; lane 0
// releases the slot on the even CTA's ring.
template <int CG>
__device__ __forceinline__ int feed_get(SharedState& ss, int i, int rank, volatile int* abort, int* err, int where) {
  const int slot = i % kTileRing;
  const uint32_t par = (i / kTileRing) & 1;
  if (!mbar_wait<CG == 2>(&ss.tile_full[slot], par, abort, err, where)) return -1;
  const int tile = *reinterpret_cast<volatile int*>(&ss.tile_ring[slot]);
  __syncwarp(__activemask());
  if (lane_id() == 0) {
    if (CG == 2 && rank != 0)
      mbar_arrive_rank(&ss.tile_empty[slot], 0);
    else
      mbar_arrive(&ss.tile_empty[slot]);
  }
  return tile;
}

// CG = 1: one CTA per SM and tile.  CG = 2: CTA pairs (clusters of two), one
// 256-row tile per pair; the even CTA issues the MMAs for both.
template <int KIND, int CG>
__global__ void __launch_bounds__(Pipe<KIND, CG>::THREADS, 1) grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr int EW = Pipe<KIND, CG>::EPI_WARPS;
  const int NST = p.nst;  // at most Pipe<KIND, CG>::STAGES (checked by the launcher)
  constexpr int SB = Pipe<KIND, CG>::STAGE_BYTES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The 128-byte-swizzled stages need a 1024-byte-aligned base; the dynamic
  // shared window of a kernel without static shared memory starts there.
  // Checked rather than padded (the padding would cost a pipeline stage's
  // worth of headroom): a misaligned base is reported, never computed on.
  // The offset is the same in every CTA, so both CTAs of a pair return here.
  if (smem_u32(smem_raw) & 1023) {
    if (threadIdx.x == 0) record_error(p.err, MOE_ERR_CUDA, 0x5A11);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* stg_base = smem + NST * SB;  // epilogue staging, Traits::EPI_BYTES per epilogue warp
  // Direct epilogue stores need no staging: the state follows the ring.
  SharedState& ss = *reinterpret_cast<SharedState*>(stg_base + (p.epi_direct ? 0 : EW * Traits<KIND>::EPI_BYTES));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = CG == 2 ? static_cast<int>(cluster_ctarank()) : 0;

  if (threadIdx.x == 0) {
    init_gemm_barriers<CG, EW>(ss);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(&ss.tmem_base, kTmemCols);
    tmem_relinquish<CG>();
  }
  build_segments<KIND, CG>(p, ss);
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the peer's barriers exist before anything arrives on them
  tc_fence_after();
  // The set-up above overlaps the previous kernel's last wave: it reads only
  // the routing tables, which are complete before the previous kernel may
  // have let this one start.  Everything below may read that kernel's output.
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tmem = ss.tmem_base;
  const int total = ss.total_tiles;
  volatile int* abort = &ss.abort;
  const int where0 = (KIND + 1) << 24 | rank << 23;

  // Ragged-K kinds take tiles from the ticket counter; the others keep the
  // static round-robin, whose fixed spread of neighbouring tiles (which share
  // operand tiles) over the CTAs measured 3-6% faster for equal-length tiles.
  constexpr bool DYN = Traits<KIND>::RAGGED_K;
  const int first = CG == 2 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int step = CG == 2 ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  const int wfeed = where0 | (6 << 20);
  // The i-th tile of this CTA (-1: none left) for every role but the ticket
  // taker.
  auto tile_of = [&](int i, int where) {
    if constexpr (DYN) {
      return feed_get<CG>(ss, i, rank, abort, p.err, where);
    } else {
      const int t = first + i * step;
      return (t < total && !*abort) ? t : -1;
    }
  };
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.tmA0);
      tma_prefetch_desc(&p.tmB0);
      ProducerState ps;
      if (DYN && rank == 0) {
        // Ticket taker: the next ticket is drawn while the current tile's
        // loads are issued, so the atomic's round trip is off the path.
        int* ctr = p.err + kErrSchedWord + 2 * KIND;
        int next = atomicAdd(ctr, 1);
        for (int i = 0;; ++i) {
          const int tile = (next < total && !*abort) ? next : -1;
          if (tile >= 0) next = atomicAdd(ctr, 1);
          if (!feed_put<CG>(ss, i, tile, abort, p.err, wfeed | (i & 0xfffff)) || tile < 0) break;
          if (p.prefetch_kb > 0 && next < total)
            prefetch_tile<KIND, CG>(p, decode_tile<KIND, CG>(p, ss, next, rank), rank);
          if (!produce_tile<KIND, CG>(p, decode_tile<KIND, CG>(p, ss, tile, rank), ss, smem, ps, abort,
                                       where0 | tile, NST, rank))
            break;
        }
        // The last ticket taker to finish sets the counters back to 0 for
        // the next launch (every taker has drawn its final ticket by then).
        const int takers = static_cast<int>(gridDim.x) / CG;
        if (atomicAdd(ctr + 1, 1) == takers - 1) {
          atomicExch(ctr, 0);
          atomicExch(ctr + 1, 0);
        }
      } else {
        for (int i = 0;; ++i) {
          const int tile = tile_of(i, wfeed | (i & 0xfffff));
          if (tile < 0) break;
          if (!DYN && p.prefetch_kb > 0 && tile + step < total)
            prefetch_tile<KIND, CG>(p, decode_tile<KIND, CG>(p, ss, tile + step, rank), rank);
          if (!produce_tile<KIND, CG>(p, decode_tile<KIND, CG>(p, ss, tile, rank), ss, smem, ps, abort,
                                       where0 | tile, NST, rank))
            break;
        }
      }
      if (*abort) producer_drain(ss, ps);
    }
  } else if (warp == 1) {
    MmaState ms;
    for (int i = 0;; ++i) {
      const int tile = tile_of(i, wfeed | (1 << 19) | (i & 0x7ffff));
      if (tile < 0 || !mma_tile<KIND, CG>(p, decode_tile<KIND, CG>(p, ss, tile, rank), ss, smem, tmem, ms,
                                          abort, where0 | (2 << 20) | tile, NST, rank))
        break;
    }
    if (*abort) mma_drain<CG>(ss, ms);
  } else {
    EpiState es;
    uint8_t* stg = stg_base + (warp - 2) * Traits<KIND>::EPI_BYTES;
    for (int i = 0;; ++i) {
      const int tile = tile_of(i, wfeed | (2 << 19) | (i & 0x7ffff));
      if (tile < 0 || !epilogue_step<KIND, CG, EW>(p, decode_tile<KIND, CG>(p, ss, tile, rank), ss, tmem, stg, es,
                                               abort, where0 | (4 << 20) | tile, rank))
        break;
    }
    epilogue_drain(ss, es);
  }

  tc_fence_before();
  __syncthreads();
  // No CTA of a pair leaves (or frees TMEM) while the other may still arrive
  // on its barriers or have MMAs read its shared memory.
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<CG>(tmem, kTmemCols);
}

// ------------------------------------------------------------------------
// The backward's dX, dW1/dW3 and dW2 GEMMs as one persistent launch.  dX is
// tensor-heavy and writes little; the weight-gradient kinds' short-K tiles
// write 256 KB of fp32 per tile after a few microseconds of MMAs.  Run one
// after the other, the write-heavy phase throttles the main loops of every
// SM at once; here one ticket counter hands out both kinds interleaved, so
// each SM alternates between them and the memory system sees a mix.  All
// three only read what dH (and the forward) wrote, so no tile waits on
// another.  Each output element is still produced by one tile with its fixed
// K order: the bits are those of the separate launches.
struct BwdGemmParams {
  GemmParams x, w13, w2;  // dX, dW1/dW3, dW2
};

// Ticket i -> (kind: 0 dX, 1 dW1/dW3, 2 dW2; tile of that kind).  The dX
// tiles sit at tickets floor(j * total / nX), spread over the whole range;
// the other tickets take the weight-gradient tiles segment by segment in
// the longest-first order, each segment's dW1/dW3 tiles then its dW2 tiles.
struct MixMap {
  int nX, tps13, tps2, total;
};
__device__ __forceinline__ int2 mix_decode(const MixMap& m, int i) {
  const long long NL = m.nX, span = m.total;
  auto upto = [&](long long v) { return v < 0 ? 0ll : min(NL, ((v + 1) * NL + span - 1) / span); };
  const long long c = upto(i), cp = upto(i - 1);
  if (c > cp) return make_int2(0, static_cast<int>(c - 1));
  const int pos = static_cast<int>(i - c), per = m.tps13 + m.tps2;
  const int oi = pos / per, local = pos - oi * per;
  if (local < m.tps13) return make_int2(1, oi * m.tps13 + local);
  return make_int2(2, oi * m.tps2 + (local - m.tps13));
}

constexpr int kBwdEpiBytes = Traits<kDX>::EPI_BYTES > Traits<kDW13>::EPI_BYTES
                                 ? Traits<kDX>::EPI_BYTES
                                 : (Traits<kDW13>::EPI_BYTES > Traits<kDW2>::EPI_BYTES ? Traits<kDW13>::EPI_BYTES
                                                                                        : Traits<kDW2>::EPI_BYTES);
template <int CG>
constexpr int bwd_gemms_smem_bytes() {
  return Pipe<kDX, CG>::STAGES * Pipe<kDX, CG>::STAGE_BYTES + kEpiWarps * kBwdEpiBytes +
         3 * static_cast<int>(sizeof(SharedState));
}
constexpr int kMixSched = 6;  // scheduling words of the error region: after the six kinds'

template <int CG>
__global__ void __launch_bounds__(kThreads, 1) bwd_gemms_kernel(const __grid_constant__ BwdGemmParams bp) {
  static_assert(Pipe<kDX, CG>::STAGE_BYTES == Pipe<kDW13, CG>::STAGE_BYTES &&
                    Pipe<kDX, CG>::STAGE_BYTES == Pipe<kDW2, CG>::STAGE_BYTES,
                "the three kinds share the ring");
  constexpr int SB = Pipe<kDX, CG>::STAGE_BYTES;
  const int NST = bp.x.nst;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  int* err = bp.x.err;
  if (smem_u32(smem_raw) & 1023) {
    if (threadIdx.x == 0) record_error(err, MOE_ERR_CUDA, 0x5A11);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* stg_base = smem + NST * SB;
  SharedState* tables = reinterpret_cast<SharedState*>(stg_base + kEpiWarps * kBwdEpiBytes);
  SharedState& ss = tables[0];   // barriers and the dX segment table
  SharedState& s13 = tables[1];  // weight-gradient tables (segment order, tiles per segment)
  SharedState& s2 = tables[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = CG == 2 ? static_cast<int>(cluster_ctarank()) : 0;

  if (threadIdx.x == 0) {
    init_gemm_barriers<CG, kEpiWarps>(ss);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(&ss.tmem_base, kTmemCols);
    tmem_relinquish<CG>();
  }
  build_segments<kDX, CG>(bp.x, ss);
  build_segments<kDW13, CG>(bp.w13, s13);
  build_segments<kDW2, CG>(bp.w2, s2);
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = ss.tmem_base;
  MixMap mm;
  mm.nX = ss.total_tiles;
  mm.tps13 = s13.tiles_per_seg;
  mm.tps2 = s2.tiles_per_seg;
  mm.total = ss.total_tiles + s13.total_tiles + s2.total_tiles;
  const int total = mm.total;
  volatile int* abort = &ss.abort;
  const int where0 = (kMixSched + 1) << 24 | rank << 23;
  const int wfeed = where0 | (6 << 20);

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&bp.x.tmA0);
      tma_prefetch_desc(&bp.w13.tmA0);
      tma_prefetch_desc(&bp.w2.tmA0);
      ProducerState ps;
      auto produce = [&](int ticket) {
        const int2 kt = mix_decode(mm, ticket);
        const int where = where0 | ticket;
        if (kt.x == 0)
          return produce_tile<kDX, CG>(bp.x, decode_tile<kDX, CG>(bp.x, ss, kt.y, rank), ss, smem, ps, abort, where,
                                       NST, rank);
        if (kt.x == 1)
          return produce_tile<kDW13, CG>(bp.w13, decode_tile<kDW13, CG>(bp.w13, s13, kt.y, rank), ss, smem, ps,
                                         abort, where, NST, rank);
        return produce_tile<kDW2, CG>(bp.w2, decode_tile<kDW2, CG>(bp.w2, s2, kt.y, rank), ss, smem, ps, abort,
                                      where, NST, rank);
      };
      if (rank == 0) {
        int* ctr = err + kErrSchedWord + 2 * kMixSched;
        int next = atomicAdd(ctr, 1);
        for (int i = 0;; ++i) {
          const int tile = (next < total && !*abort) ? next : -1;
          if (tile >= 0) next = atomicAdd(ctr, 1);
          if (!feed_put<CG>(ss, i, tile, abort, err, wfeed | (i & 0xfffff)) || tile < 0) break;
          if (!produce(tile)) break;
        }
        const int takers = static_cast<int>(gridDim.x) / CG;
        if (atomicAdd(ctr + 1, 1) == takers - 1) {
          atomicExch(ctr, 0);
          atomicExch(ctr + 1, 0);
        }
      } else {
        for (int i = 0;; ++i) {
          const int tile = feed_get<CG>(ss, i, rank, abort, err, wfeed | (i & 0xfffff));
          if (tile < 0 || !produce(tile)) break;
        }
      }
      if (*abort) producer_drain(ss, ps);
    }
  } else if (warp == 1) {
    MmaState ms;
    for (int i = 0;; ++i) {
      const int tile = feed_get<CG>(ss, i, rank, abort, err, wfeed | (1 << 19) | (i & 0x7ffff));
      if (tile < 0) break;
      const int2 kt = mix_decode(mm, tile);
      const int where = where0 | (2 << 20) | tile;
      bool ok;
      if (kt.x == 0)
        ok = mma_tile<kDX, CG>(bp.x, decode_tile<kDX, CG>(bp.x, ss, kt.y, rank), ss, smem, tmem, ms, abort, where,
                               NST, rank);
      else if (kt.x == 1)
        ok = mma_tile<kDW13, CG>(bp.w13, decode_tile<kDW13, CG>(bp.w13, s13, kt.y, rank), ss, smem, tmem, ms, abort,
                                 where, NST, rank);
      else
        ok = mma_tile<kDW2, CG>(bp.w2, decode_tile<kDW2, CG>(bp.w2, s2, kt.y, rank), ss, smem, tmem, ms, abort,
                                where, NST, rank);
      if (!ok) break;
    }
    if (*abort) mma_drain<CG>(ss, ms);
  } else {
    EpiState es;
    uint8_t* stg = stg_base + (warp - 2) * kBwdEpiBytes;
    for (int i = 0;; ++i) {
      const int tile = feed_get<CG>(ss, i, rank, abort, err, wfeed | (2 << 19) | (i & 0x7ffff));
      if (tile < 0) break;
      const int2 kt = mix_decode(mm, tile);
      const int where = where0 | (4 << 20) | tile;
      bool ok;
      if (kt.x == 0)
        ok = epilogue_step<kDX, CG>(bp.x, decode_tile<kDX, CG>(bp.x, ss, kt.y, rank), ss, tmem, stg, es, abort, where,
                                    rank);
      else if (kt.x == 1)
        ok = epilogue_step<kDW13, CG>(bp.w13, decode_tile<kDW13, CG>(bp.w13, s13, kt.y, rank), ss, tmem, stg, es,
                                      abort, where, rank);
      else
        ok = epilogue_step<kDW2, CG>(bp.w2, decode_tile<kDW2, CG>(bp.w2, s2, kt.y, rank), ss, tmem, stg, es, abort,
                                     where, rank);
      if (!ok) break;
    }
    epilogue_drain(ss, es);
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<CG>(tmem, kTmemCols);
}

// Kinds that run on CTA pairs (bit = GemmKind): measured at the 8192-token
// DeepSeek-V2-Lite-like shape, pairs win for all six (moe_autotune re-decides
// per layer).
int g_pair_kinds = (1 << 6) - 1;
int g_prefetch_kb[6] = {0, 0, 0, 0, 0, 0};  // per kind: next-tile K blocks prefetched into L2
int g_tile_order[6] = {0, 0, 0, 0, 0, 0};   // per ragged-K kind: 0 longest first, 1 long tiles interleaved
int g_stages[6] = {0, 0, 0, 0, 0, 0};       // per kind: pipeline stages (0: as many as fit)
int g_epi_direct[6] = {0, 0, 0, 0, 0, 0};   // per fp32-output kind: 1 = unstaged epilogue stores

// Launch configuration of one kind; CG = 2 adds the cluster dimension.
template <int KIND, int CG>
void launch_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, cudaStream_t s) {
  cfg = {};
  cfg.blockDim = dim3(Pipe<KIND, CG>::THREADS);
  cfg.dynamicSmemBytes = launch_smem_bytes<KIND, CG>();
  cfg.stream = s;
  if constexpr (CG == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
}

// Number of CTA pairs of kind KIND that can be resident at once (cached).
template <int KIND>
int pair_capacity() {
  static int cached = 0;
  if (cached == 0) {
    auto kern = grouped_gemm_kernel<KIND, 2>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, launch_smem_bytes<KIND, 2>()) !=
        cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    launch_config<KIND, 2>(cfg, attr, nullptr);
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return 0;
    cached = n;
  }
  return cached;
}

template <int KIND, int CG>
int launch_kind(const GemmArgs& a, cudaStream_t s, int grid_override) {
  GemmParams p;
  if (!fill_params<KIND, CG>(a, p)) return MOE_ERR_CUDA;
  p.prefetch_kb = g_prefetch_kb[KIND];
  p.tile_order = g_tile_order[KIND];
  p.epi_direct = g_epi_direct[KIND];
  // Fewer stages leave part of the ring unused; the launch still takes the
  // whole shared-memory budget, so one CTA per SM stays resident.
  const int max_st = p.epi_direct ? direct_stages<KIND, CG>() : Pipe<KIND, CG>::STAGES;
  p.nst = (g_stages[KIND] >= 2 && g_stages[KIND] < max_st) ? g_stages[KIND] : max_st;
  constexpr int kSmem = launch_smem_bytes<KIND, CG>();
  static_assert(kSmem <= kSmemBudget, "shared memory budget of one CTA");
  static_assert(direct_stages<KIND, CG>() <= kMaxStages, "stage barriers");
  auto kern = grouped_gemm_kernel<KIND, CG>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return MOE_ERR_CUDA;
  int grid = grid_override > 0 ? grid_override : num_sms();
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  launch_config<KIND, CG>(cfg, attr, s);
  set_pdl_attr(attr[cfg.numAttrs]);
  cfg.attrs = attr;
  ++cfg.numAttrs;
  if constexpr (CG == 2) {
    // Persistent: only as many pairs as can be resident at once (an SM
    // left without a partner stays idle rather than adding a second wave).
    const int max_pairs = pair_capacity<KIND>();
    if (max_pairs <= 0) return MOE_ERR_CUDA;
    grid = 2 * std::max(1, std::min(max_pairs, grid / 2));
  }
  cfg.gridDim = dim3(grid);
  constexpr int kTrace[6] = {MOE_K_GEMM1, MOE_K_GEMM2, MOE_K_GEMM_DH, MOE_K_GEMM_DX, MOE_K_GEMM_DW13, MOE_K_GEMM_DW2};
  TraceScope trace_scope(kTrace[KIND], s);
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int CG>
int launch_bwd_gemms_cg(const GemmArgs& a, cudaStream_t s, int grid_override) {
  BwdGemmParams bp;
  std::memset(&bp, 0, sizeof(bp));
  if (!fill_params<kDX, CG>(a, bp.x) || !fill_params<kDW13, CG>(a, bp.w13) || !fill_params<kDW2, CG>(a, bp.w2))
    return MOE_ERR_CUDA;
  bp.x.nst = bp.w13.nst = bp.w2.nst = Pipe<kDX, CG>::STAGES;
  constexpr int kSmem = bwd_gemms_smem_bytes<CG>();
  static_assert(kSmem <= 232448, "shared memory budget of one CTA");
  auto kern = bwd_gemms_kernel<CG>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  int grid = grid_override > 0 ? grid_override : num_sms();
  if constexpr (CG == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static int cap = 0;
    if (cap == 0) {
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3(2 * (num_sms() / 2));
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n <= 0) return MOE_ERR_CUDA;
      cap = n;
    }
    grid = 2 * std::max(1, std::min(cap, grid / 2));
  }
  cfg.gridDim = dim3(grid);
  TraceScope trace_scope(MOE_K_BWD_GEMMS, s);
  if (cudaLaunchKernelEx(&cfg, kern, bp) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int KIND>
int launch_any(const GemmArgs& a, cudaStream_t s, int grid_override) {
  return (g_pair_kinds >> KIND) & 1 ? launch_kind<KIND, 2>(a, s, grid_override)
                                    : launch_kind<KIND, 1>(a, s, grid_override);
}

}  // namespace

int launch_gemm(GemmKind kind, const GemmArgs& a, cudaStream_t s, int grid_override) {
  switch (kind) {
    case kG1: return launch_any<kG1>(a, s, grid_override);
    case kG2: return launch_any<kG2>(a, s, grid_override);
    case kDH: return launch_any<kDH>(a, s, grid_override);
    case kDX: return launch_any<kDX>(a, s, grid_override);
    case kDW13: return launch_any<kDW13>(a, s, grid_override);
    case kDW2: return launch_any<kDW2>(a, s, grid_override);
  }
  return MOE_ERR_ARG;
}

int launch_bwd_gemms(const GemmArgs& a, cudaStream_t s, int grid_override) {
  const bool pairs = ((g_pair_kinds >> kDX) & 1) && ((g_pair_kinds >> kDW13) & 1) && ((g_pair_kinds >> kDW2) & 1);
  return pairs ? launch_bwd_gemms_cg<2>(a, s, grid_override) : launch_bwd_gemms_cg<1>(a, s, grid_override);
}

int gemm_pair_capacity(GemmKind kind) {
  switch (kind) {
    case kG1: return pair_capacity<kG1>();
    case kG2: return pair_capacity<kG2>();
    case kDH: return pair_capacity<kDH>();
    case kDX: return pair_capacity<kDX>();
    case kDW13: return pair_capacity<kDW13>();
    case kDW2: return pair_capacity<kDW2>();
  }
  return 0;
}

int set_gemm_prefetch(GemmKind kind, int kblocks) {
  if (kind < kG1 || kind > kDW2) return -1;
  const int prev = g_prefetch_kb[kind];
  g_prefetch_kb[kind] = kblocks < 0 ? 0 : (kblocks > 64 ? 64 : kblocks);
  return prev;
}

int set_gemm_tile_order(GemmKind kind, int order) {
  if (kind != kDW13 && kind != kDW2) return -1;
  const int prev = g_tile_order[kind];
  g_tile_order[kind] = order ? 1 : 0;
  return prev;
}

int set_gemm_epilogue(GemmKind kind, int direct) {
  if (kind != kG2 && kind != kDX && kind != kDW13 && kind != kDW2) return -1;
  const int prev = g_epi_direct[kind];
  g_epi_direct[kind] = direct ? 1 : 0;
  return prev;
}

int set_gemm_stages(GemmKind kind, int stages) {
  if (kind < kG1 || kind > kDW2) return -1;
  const int prev = g_stages[kind];
  g_stages[kind] = stages < 0 ? 0 : stages;
  return prev;
}

template <int KIND>
int max_stages_of(int cta_group, bool direct) {
  if (cta_group == 2) return direct ? direct_stages<KIND, 2>() : Pipe<KIND, 2>::STAGES;
  return direct ? direct_stages<KIND, 1>() : Pipe<KIND, 1>::STAGES;
}

int gemm_max_stages(GemmKind kind, int cta_group, int direct) {
  switch (kind) {
    case kG1: return max_stages_of<kG1>(cta_group, false);
    case kG2: return max_stages_of<kG2>(cta_group, direct != 0);
    case kDH: return max_stages_of<kDH>(cta_group, false);
    case kDX: return max_stages_of<kDX>(cta_group, direct != 0);
    case kDW13: return max_stages_of<kDW13>(cta_group, direct != 0);
    case kDW2: return max_stages_of<kDW2>(cta_group, direct != 0);
  }
  return 0;
}

int gemm_max_stages(GemmKind kind, int cta_group) {
  return kind >= kG1 && kind <= kDW2 ? gemm_max_stages(kind, cta_group, g_epi_direct[kind]) : 0;
}

int gemm_pair_kinds() { return g_pair_kinds; }

int set_gemm_pair_kinds(int mask) {
  const int prev = g_pair_kinds;
  g_pair_kinds = mask & ((1 << 6) - 1);
  return prev;
}

}  // namespace moe

// MegaKernels: one persistent launch for
//   forward:  dispatch gather -> GEMM 1 (+SiLU*mul) -> GEMM 2 (+routing
//             weight) -> combine;
//   backward input part:  combine-bwd gather (G = dy rows) -> dH GEMM
//             (+SwiGLU backward, dw partials) -> dX GEMM -> slot-order dx sum.
// Both have the same shape (a row gather, a first grouped GEMM over those
// rows, a second grouped GEMM over the first one's row blocks, a per-token
// fp32 sum of the second one's rows), so one kernel template serves both.
//
// UniEP page ("Unified Expert-Parallel MoE MegaKernel for LLM Training"),
// section 2.2: exactly one persistent worker per SM, roles chosen at run time
// from a ticket taken off one global atomic counter (the linearised task
// space puts communication tasks first, compute tasks after), and a
// global-memory scoreboard that marks when every token of a GroupGEMM tile
// has arrived, which compute workers poll before starting the tile.  On one
// GPU the communication task is the local dispatch gather; the scoreboard is
// a set of readiness counters (A, B: the first and second GEMM):
//   ctr[0]                   ticket cursor
//   ctr[1]                   B warp-tiles finished (the token sums wait on all)
//   ctr[2]                   sum cursor: after the last ticket every warp of
//                            every CTA claims tokens one at a time from it
//   ctr[3]                   gather parts finished (NG * CG: every block is in)
//   ctr[kCtrXp + g]          gathered row block g (mp.grows rows) written
//   ctr[kCtrXp + NG + mt]    A warp-tiles finished of m-tile mt
//                            (B tiles of mt wait for all of them)
// The UniEP page (section 2.2) has its MegaKernels serve the backward steps
// too; the backward one here is its input-gradient (B) part.
// A task only ever waits on tasks with lower tickets, and each CTA runs its
// tasks in ticket order, so the lowest unfinished task can always proceed:
// no deadlock, with or without co-residency of all CTAs.  Every wait is
// bounded (1 s) and reports MOE_ERR_TIMEOUT instead of hanging.
//
// GEMM tiles run exactly the MMA sequence and epilogue of the stand-alone
// grouped GEMM kernels and the token sums add in the same order as the
// stand-alone sum kernel, so the outputs are bitwise equal to the unfused
// chain.
#include <algorithm>

#include "gemm_tiles.cuh"

namespace moe {
namespace {

constexpr int kTq = 4;              // depth of the producer -> consumer task FIFO

constexpr int kCtrXp = 8;
constexpr int kMaxTokRows = 12;     // k <= 8 routed + S <= 4 shared rows per token
constexpr int kMaxMegaStages = kMaxStages;

struct MegaParams {
  GemmParams g1, g2;           // first (A) and second (B) grouped GEMM
  const uint16_t* x;           // gather source rows (x forward, dy backward)
  const int32_t* row_token;
  const int32_t* dest;
  uint16_t* Xp;                // gathered rows (Xp forward, G backward)
  const float* Op;             // rows summed per token (O' forward, dXp backward)
  float* y;                    // token sums (y forward, dx backward)
  int* ctr;
  int NG;
  int grows;  // gathered rows per gather task (kMegaGatherRows or 128)
  int skip;  // testing aid: ticket treated as never done (-1: none)
  // optional per-task timeline: records_per_cta records of 3 x u64
  // (ticket | role << 32 | cta << 40, start ns, end ns) per CTA, the first
  // half for the producer, the second for the first epilogue warp
  unsigned long long* trace;
  int trace_per_cta;
};

int g_skip_ticket = -1;
unsigned long long* g_trace_buf = nullptr;
int g_trace_per_cta = 0;

__device__ __forceinline__ void trace_record(const MegaParams& mp, int role, int& n, int id, uint64_t t0) {
  if (!mp.trace) return;
  const int half = mp.trace_per_cta / 2;
  if (n >= half) return;
  unsigned long long* r =
      mp.trace + 3ull * (static_cast<size_t>(blockIdx.x) * mp.trace_per_cta + static_cast<size_t>(role) * half + n);
  r[0] = static_cast<unsigned long long>(static_cast<unsigned>(id)) | (static_cast<unsigned long long>(role) << 32) |
         (static_cast<unsigned long long>(blockIdx.x) << 40);
  r[1] = t0;
  r[2] = globaltimer_ns();
  ++n;
}

// Shapes of one MegaKernel: its two GEMM kinds, its pipeline depth and its
// CTA group.  One CTA per tile: 4 stages of 48 KB.  CTA pairs (256-row
// tiles, tcgen05 CTA group of two, as the stand-alone grouped GEMMs run by
// default): 6 stages of 32 KB.  Both fit beside the larger of the two
// kinds' epilogue staging (GEMM 1: 6 KB a warp, dH: 8 KB).
template <int KA, int KB, int NST, int CG = 1>
struct Mega {
  static constexpr int STAGES = NST;
  static constexpr int STAGE_BYTES = Pipe<KA, CG>::STAGE_BYTES;
  static_assert(Pipe<KA, CG>::STAGE_BYTES == Pipe<KB, CG>::STAGE_BYTES, "both GEMMs share the ring");
  // epilogue staging per warp: the larger of the two kinds'
  static constexpr int EPI_BYTES =
      Traits<KA>::EPI_BYTES > Traits<KB>::EPI_BYTES ? Traits<KA>::EPI_BYTES : Traits<KB>::EPI_BYTES;
};

// Token sums after the GEMMs: each warp stages the rows of one (token,
// column span) unit in its own 32 KB of the then idle pipeline ring.
constexpr int kSumWarps = kThreads / 32;
constexpr int kSumBytes = 32 * 1024;

struct MegaShared {
  SharedState g;
  uint64_t tq_full[kTq], tq_empty[kTq], gbar[kMaxMegaStages], sbar[kSumWarps];
  int tq[kTq];
  int ntn1, ntn2, nt1, nt2, total;
};

template <int KA, int KB, int NST, int CG = 1>
constexpr int mega_smem_bytes() {
  return NST * Mega<KA, KB, NST, CG>::STAGE_BYTES + kEpiWarps * Mega<KA, KB, NST, CG>::EPI_BYTES +
         static_cast<int>(sizeof(MegaShared));
}
static_assert(mega_smem_bytes<kG1, kG2, 4>() <= 232448, "shared memory budget of one CTA");
static_assert(mega_smem_bytes<kDH, kDX, 4>() <= 232448, "shared memory budget of one CTA");
static_assert(mega_smem_bytes<kG1, kG2, 6, 2>() <= 232448, "shared memory budget of one CTA");
static_assert(mega_smem_bytes<kDH, kDX, 6, 2>() <= 232448, "shared memory budget of one CTA");
// the token sums' staging fits the ring and epilogue staging of every shape
template <int KA, int KB, int NST, int CG>
constexpr bool sum_staging_fits() {
  return NST * Mega<KA, KB, NST, CG>::STAGE_BYTES + kEpiWarps * Mega<KA, KB, NST, CG>::EPI_BYTES >=
         kSumWarps * kSumBytes;
}
static_assert(sum_staging_fits<kG1, kG2, 4, 1>() && sum_staging_fits<kDH, kDX, 4, 1>() &&
                  sum_staging_fits<kG1, kG2, 6, 2>() && sum_staging_fits<kDH, kDX, 6, 2>(),
              "token-sum staging");

// Bounded acquire-spin until *c >= target.
__device__ bool wait_counter(const int* c, int target, volatile int* abort, int* err, int where) {
  if (ld_acquire_gpu(c) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu(c) < target) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_error(err, MOE_ERR_TIMEOUT_CODE, where);
      *abort = 1;
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Publishes this warp's global stores -- its TMA stores (completed first)
// and any direct stores -- to other CTAs, including their TMA reads, then
// lane 0 adds one to the readiness counter.
__device__ __forceinline__ void warp_signal(int* counter) {
  if ((threadIdx.x & 31) == 0) bulk_wait_all();
  fence_proxy_async_global();
  __threadfence();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) red_release_gpu_add(counter, 1);
}

// Gather task g (producer lane): gathered rows [grows*g, grows*(g+1)) <-
// source[row_token], a bulk load per row into the stage buffers (up to
// NST-1 chunks in flight) and one bulk store per chunk (its destination rows
// are consecutive), then publish the block.
struct GatherState {
  uint32_t par = 0;      // next wait parity of gbar[b] (bit b)
  uint32_t pending = 0;  // buffers with loads issued but not yet waited on
};

// With CTA pairs each CTA of the pair gathers its half of the block (`part`
// of `nparts`) and signals the block's counter once (a block is complete
// at nparts signals).
template <int NST, int SB>
__device__ bool gather_task(const MegaParams& mp, MegaShared& ms, uint8_t* smem, int g, GatherState& gs,
                            volatile int* abort, int where, int part = 0, int nparts = 1) {
  const int d = mp.g1.d;
  const uint32_t rb = 2u * d;
  const int rps = min(mp.grows, SB / static_cast<int>(rb));  // >= 1: checked on the host
  const int blk0 = g * mp.grows;
  const int blk_rows = min(mp.grows, mp.g1.R - blk0);
  const int per = (blk_rows + nparts - 1) / nparts;
  const int r0 = blk0 + min(blk_rows, part * per);
  const int nrows = min(blk_rows, (part + 1) * per) - min(blk_rows, part * per);
  const int nchunk = (nrows + rps - 1) / rps;
  for (int c = 0; c <= nchunk; ++c) {
    if (c < nchunk) {
      const int b = c % NST;
      if (c >= NST) bulk_wait_read<NST - 2>();  // chunk c-NST finished reading buffer b
      const int n = min(rps, nrows - c * rps);
      uint8_t* buf = smem + b * SB;
      mbar_arrive_expect_tx(&ms.gbar[b], n * rb);
      for (int i = 0; i < n; ++i) {
        int tok = mp.row_token[r0 + c * rps + i];
        if (!debug_ok(static_cast<unsigned>(tok) < static_cast<unsigned>(mp.g1.T), mp.g1.err, kDbgMegaGather,
                      r0 + c * rps + i))
          tok = 0;
        bulk_load(buf + i * rb, mp.x + static_cast<size_t>(tok) * d, rb, &ms.gbar[b]);
      }
      gs.pending |= 1u << b;
    }
    if (c > 0) {
      const int pc = c - 1, b = pc % NST;
      if (!mbar_wait(&ms.gbar[b], (gs.par >> b) & 1, abort, mp.g1.err, where)) return false;
      gs.par ^= 1u << b;
      gs.pending &= ~(1u << b);
      const int n = min(rps, nrows - pc * rps);
      uint8_t* buf = smem + b * SB;
      // the chunk's destination rows are consecutive: one bulk store
      bulk_store(mp.Xp + static_cast<size_t>(r0 + pc * rps) * d, buf, n * rb);
      bulk_commit();
    }
  }
  bulk_wait_all();
  fence_proxy_async_global();
  red_release_gpu_add(&mp.ctr[kCtrXp + g], 1);
  red_release_gpu_add(&mp.ctr[3], 1);
  return true;
}

__device__ void gather_drain(MegaShared& ms, const GatherState& gs) {
  bulk_wait_all();
  for (int b = 0; b < kMaxMegaStages; ++b)
    if (gs.pending & (1u << b)) mbar_wait_drain(&ms.gbar[b], (gs.par >> b) & 1);
}

// Tile t2 of the second GEMM described with the first one's segment table
// (both run over the same rows, so they share m-tiles).
template <int KA, int KB, int CG = 1>
__device__ __forceinline__ TileInfo decode_g2(const MegaParams& mp, const MegaShared& ms, int t2, int rank = 0) {
  const int mt = t2 / ms.ntn2, nb = t2 - mt * ms.ntn2;
  TileInfo t = decode_tile<KA, CG>(mp.g1, ms.g, mt * ms.ntn1, rank);
  t.n0 = nb * Traits<KB>::BNE;
  t.nkb = mp.g2.K / kBK;
  return t;
}

// Token sums, run by every warp of every CTA once its part of the ticket
// space is done and all second-GEMM tiles are published: warps claim units
// of one token and one column span from their own cursor (ctr[2]) until
// none are left.  A unit's rows (the token's k routed rows by dest, then its
// shared rows) are brought into the warp's 32 KB of shared memory with one
// bulk copy each -- with a handful of warps per SM, loads straight into
// registers leave too few bytes in flight to stream at HBM rate -- and are
// summed in slot order in fp32, the same order as the stand-alone sum
// kernel, so the bits are the same.
__device__ void combine_phase(const MegaParams& mp, int nt2, int cg, uint8_t* smem, MegaShared& ms,
                              volatile int* abort, int* err) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ok = 1;
  if (lane == 0) {
    ok = wait_counter(&mp.ctr[1], kEpiWarps * cg * nt2, abort, err, (0x0F << 24) | (5 << 20)) ? 1 : 0;
    __threadfence();
  }
  if (!__shfl_sync(0xffffffffu, ok, 0)) return;
  const int T = mp.g1.T, k = mp.g1.k, S = mp.g1.S, R = mp.g1.R, d = mp.g1.d;
  const int nr = k + S;
  // span: columns per unit, a multiple of 64 floats whose nr rows fit the buffer
  const int W = min(d, (kSumBytes / (4 * nr)) / 64 * 64);
  const int nspan = (d + W - 1) / W;
  const long long units = static_cast<long long>(T) * nspan;
  float* buf = reinterpret_cast<float*>(smem + warp * kSumBytes);
  uint64_t* bar = &ms.sbar[warp];
  uint32_t par = 0;
  int next = 0;
  if (lane == 0) next = atomicAdd(&mp.ctr[2], 1);
  while (true) {
    int u = __shfl_sync(0xffffffffu, next, 0);
    if (u >= units) break;
    if (lane == 0) next = atomicAdd(&mp.ctr[2], 1);  // the next claim's round trip overlaps this unit
    const int t = u / nspan, c0 = (u - t * nspan) * W;
    const int cols = min(W, d - c0);
    long long myrow = 0;
    if (lane < k) {
      myrow = mp.dest[static_cast<size_t>(t) * k + lane];
      if (!debug_ok(myrow >= 0 && myrow < R, err, kDbgMegaCombine, t)) myrow = 0;
    } else if (lane < nr) {
      myrow = R + static_cast<long long>(lane - k) * T + t;
    }
    // the buffer's previous reads (generic proxy) before the copies refill it
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nr * cols * 4));
    __syncwarp();
    if (lane < nr)
      bulk_load(buf + lane * W, mp.Op + myrow * d + c0, static_cast<uint32_t>(cols * 4), bar);
    if (!mbar_wait(bar, par, abort, err, (0x0F << 24) | (6 << 20) | (t & 0xFFFFF))) return;
    par ^= 1;
    const float4* rows4 = reinterpret_cast<const float4*>(buf);
    float4* o = reinterpret_cast<float4*>(mp.y + static_cast<size_t>(t) * d + c0);
    const int nv = cols / 4, wv = W / 4;
    for (int v = lane; v < nv; v += 32) {
      float4 acc = rows4[v];
      for (int j = 1; j < nr; ++j) {
        const float4 x = rows4[j * wv + v];
        acc.x += x.x;
        acc.y += x.y;
        acc.z += x.z;
        acc.w += x.w;
      }
      o[v] = acc;
    }
  }
}

// Task FIFO of a CTA pair: the even CTA's producer claims each ticket and
// writes it to both CTAs' rings; every other role of both CTAs (the odd
// CTA's producer too) reads it and releases the slot on the even CTA's ring.
template <int CG>
__device__ __forceinline__ bool tq_put(MegaShared& ms, int slot, int id) {
  ms.tq[slot] = id;
  if constexpr (CG == 2) {
    st_shared_rank(&ms.tq[slot], 1, id);
    mbar_arrive_rank(&ms.tq_full[slot], 1);  // release at cluster scope: the store above is seen first
  }
  mbar_arrive(&ms.tq_full[slot]);
  return true;
}
template <int CG>
__device__ __forceinline__ int tq_get(MegaShared& ms, int slot, uint32_t par, int rank, volatile int* abort, int* err,
                                      int where, bool* ok) {
  *ok = mbar_wait<CG == 2>(&ms.tq_full[slot], par, abort, err, where);
  if (!*ok) return 0;
  const int id = *reinterpret_cast<volatile int*>(&ms.tq[slot]);
  __syncwarp(__activemask());
  if (lane_id() == 0) {
    if (CG == 2 && rank != 0)
      mbar_arrive_rank(&ms.tq_empty[slot], 0);
    else
      mbar_arrive(&ms.tq_empty[slot]);
  }
  return id;
}

template <int KA, int KB, int NST, int CG>
__global__ void __launch_bounds__(kThreads, 1) mega_kernel(const __grid_constant__ MegaParams mp) {
  constexpr int EPI = Mega<KA, KB, NST, CG>::EPI_BYTES;
  constexpr int SB = Mega<KA, KB, NST, CG>::STAGE_BYTES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // see grouped_gemm_kernel: checked, not padded
    if (threadIdx.x == 0) record_error(mp.g1.err, MOE_ERR_CUDA, 0x5A11);
    return;
  }
  uint8_t* smem = smem_raw;
  MegaShared& ms = *reinterpret_cast<MegaShared*>(smem + NST * SB + kEpiWarps * EPI);
  SharedState& ss = ms.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = CG == 2 ? static_cast<int>(cluster_ctarank()) : 0;
  int* err = mp.g1.err;

  if (threadIdx.x == 0) {
    init_gemm_barriers<CG>(ss);
    for (int q = 0; q < kTq; ++q) {
      mbar_init(&ms.tq_full[q], 1);
      // readers of a slot: MMA warp + epilogue warps (of both CTAs of a pair,
      // plus the odd CTA's producer)
      mbar_init(&ms.tq_empty[q], CG == 2 ? 2 * (1 + kEpiWarps) + 1 : 1 + kEpiWarps);
    }
    for (int b = 0; b < NST; ++b) mbar_init(&ms.gbar[b], 1);
    for (int w = 0; w < kSumWarps; ++w) mbar_init(&ms.sbar[w], 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(&ss.tmem_base, kTmemCols);
    tmem_relinquish<CG>();
  }
  build_segments<KA, CG>(mp.g1, ss);
  if (threadIdx.x == 0) {
    ms.ntn1 = (mp.g1.N + Traits<KA>::BNE - 1) / Traits<KA>::BNE;
    ms.ntn2 = (mp.g2.N + Traits<KB>::BNE - 1) / Traits<KB>::BNE;
    ms.nt1 = ss.total_tiles;
    ms.nt2 = (ms.nt1 / ms.ntn1) * ms.ntn2;
    ms.total = mp.NG + ms.nt1 + ms.nt2;  // combine is claimed per token afterwards
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the peer's barriers exist before anything arrives on them
  tc_fence_after();
  const uint32_t tmem = ss.tmem_base;
  volatile int* abort = &ss.abort;
  const int NG = mp.NG, nt1 = ms.nt1, nt2 = ms.nt2, total = ms.total;
  const int e1 = NG + nt1, e2 = NG + nt1 + nt2;  // ends of the GEMM-1 and GEMM-2 ticket ranges
  constexpr int kW = 0x0F << 24;
  // signals that complete a readiness counter: one per epilogue warp of the
  // tile's CTAs (per first-GEMM n-tile for the m-tile counters)
  constexpr int kTileSignals = kEpiWarps * CG;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&mp.g1.tmA0);
      tma_prefetch_desc(&mp.g1.tmB0);
      tma_prefetch_desc(&mp.g2.tmA0);
      tma_prefetch_desc(&mp.g2.tmB0);
      ProducerState ps;
      GatherState gs;
      int slot = 0, tn = 0;
      uint32_t tph = 0;
      // The even CTA holds the next ticket while it works on the current one,
      // so the atomic's round trip is off the path between tiles (a CTA still
      // runs its tickets in increasing order).
      int next = rank == 0 ? atomicAdd(&mp.ctr[0], 1) : 0;
      bool gathered = false;  // every gather block is in: no per-block waits any more
      while (!*abort) {
        int id;
        uint64_t t_claim;
        if (rank == 0) {
          if (!mbar_wait<CG == 2>(&ms.tq_empty[slot], tph ^ 1, abort, err, kW | (1 << 20))) break;
          id = next;
          if (id < total) next = atomicAdd(&mp.ctr[0], 1);
          t_claim = globaltimer_ns();
          tq_put<CG>(ms, slot, id);
        } else {
          bool ok;
          id = tq_get<CG>(ms, slot, tph, rank, abort, err, kW | (1 << 20), &ok);
          if (!ok) break;
          t_claim = globaltimer_ns();
        }
        if (++slot == kTq) {
          slot = 0;
          tph ^= 1;
        }
        if (id >= total) break;
        if (id == mp.skip) continue;
        const int where = kW | (1 << 20) | (id & 0xFFFFF);
        if (id < NG) {
          if (!gather_task<NST, SB>(mp, ms, smem, id, gs, abort, where, rank, CG)) break;
        } else if (id < e1) {
          const TileInfo t = decode_tile<KA, CG>(mp.g1, ss, id - NG, rank);
          if (t.active && !t.shared && !gathered) {  // routed rows come from the gathered rows: wait for their blocks
            if (ld_acquire_gpu(&mp.ctr[3]) >= NG * CG) {
              gathered = true;
            } else {
              const int g0 = t.grow0 / mp.grows, g1 = (t.grow0 + t.rows - 1) / mp.grows;
              bool ok = true;
              for (int g = g0; g <= g1 && ok; ++g) ok = wait_counter(&mp.ctr[kCtrXp + g], CG, abort, err, where);
              if (!ok) break;
            }
            fence_proxy_async_global();
          }
          if (!produce_tile<KA, CG>(mp.g1, t, ss, smem, ps, abort, where, NST, rank)) break;
        } else if (id < e2) {
          const int t2 = id - e1;
          const int mt = t2 / ms.ntn2;
          if (!wait_counter(&mp.ctr[kCtrXp + NG + mt], kTileSignals * ms.ntn1, abort, err, where)) break;
          fence_proxy_async_global();
          if (!produce_tile<KB, CG>(mp.g2, decode_g2<KA, KB, CG>(mp, ms, t2, rank), ss, smem, ps, abort, where, NST,
                                    rank))
            break;
        }
        trace_record(mp, 0, tn, id, t_claim);
      }
      if (*abort) {
        producer_drain(ss, ps);
        gather_drain(ms, gs);
      }
    }
    __syncwarp();
    if (!*abort) combine_phase(mp, nt2, CG, smem, ms, abort, err);
  } else if (warp == 1) {
    MmaState mst;
    int slot = 0;
    uint32_t tph = 0;
    while (true) {
      bool ok;
      const int id = tq_get<CG>(ms, slot, tph, rank, abort, err, kW | (2 << 20), &ok);
      if (!ok) break;
      if (++slot == kTq) {
        slot = 0;
        tph ^= 1;
      }
      if (id >= total) break;
      if (id == mp.skip) continue;
      const int where = kW | (2 << 20) | (id & 0xFFFFF);
      if (id >= NG && id < e1)
        ok = mma_tile<KA, CG>(mp.g1, decode_tile<KA, CG>(mp.g1, ss, id - NG, rank), ss, smem, tmem, mst, abort, where,
                              NST, rank);
      else if (id >= e1 && id < e2)
        ok = mma_tile<KB, CG>(mp.g2, decode_g2<KA, KB, CG>(mp, ms, id - e1, rank), ss, smem, tmem, mst, abort, where,
                              NST, rank);
      if (!ok) break;
    }
    if (*abort) mma_drain<CG>(ss, mst);
    if (!*abort) combine_phase(mp, nt2, CG, smem, ms, abort, err);
  } else {
    EpiState es;
    uint8_t* stg = smem + NST * SB + (warp & 3) * EPI;
    int slot = 0, tn = 0;
    uint32_t tph = 0;
    // A tile's readiness signal waits for its stores to complete; it is sent
    // once the next task is in hand, while that tile's accumulator is still
    // being computed, so the wait is off the epilogue's path.
    int* pending = nullptr;
    while (true) {
      bool ok;
      const int id = tq_get<CG>(ms, slot, tph, rank, abort, err, kW | (3 << 20), &ok);
      if (pending) {
        warp_signal(pending);
        pending = nullptr;
      }
      if (!ok) break;
      const uint64_t t_pop = globaltimer_ns();
      if (++slot == kTq) {
        slot = 0;
        tph ^= 1;
      }
      if (id >= total) break;
      if (id == mp.skip) continue;
      const int where = kW | (3 << 20) | (id & 0xFFFFF);
      if (id >= NG && id < e1) {
        const int t1 = id - NG;
        if (!epilogue_step<KA, CG>(mp.g1, decode_tile<KA, CG>(mp.g1, ss, t1, rank), ss, tmem, stg, es, abort, where,
                                   rank))
          break;
        pending = &mp.ctr[kCtrXp + NG + t1 / ms.ntn1];
      } else if (id >= e1 && id < e2) {
        if (!epilogue_step<KB, CG>(mp.g2, decode_g2<KA, KB, CG>(mp, ms, id - e1, rank), ss, tmem, stg, es, abort,
                                   where, rank))
          break;
        pending = &mp.ctr[1];
      }
      if (warp == 2 && lane == 0) trace_record(mp, 1, tn, id, t_pop);
    }
    epilogue_drain(ss, es);
    if (!*abort) combine_phase(mp, nt2, CG, smem, ms, abort, err);
  }

  tc_fence_before();
  __syncthreads();
  // No CTA of a pair leaves (or frees TMEM) while the other may still arrive
  // on its barriers or have MMAs read its shared memory.
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<CG>(tmem, kTmemCols);
}

// Pairs of MegaKernel <KA, KB, NST, 2> resident at once (cached; 0 if the
// query fails).
template <int KA, int KB, int NST>
int mega_pair_capacity() {
  static int cached = -1;
  if (cached < 0) {
    auto kern = mega_kernel<KA, KB, NST, 2>;
    constexpr int kSmem = mega_smem_bytes<KA, KB, NST, 2>();
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1)
      n = 0;
    cached = n;
  }
  return cached;
}

// Launches MegaKernel <KA, KB, NST, CG> with the two GEMMs' arguments `a`
// (filled for both kinds), the gather (src rows by row_token into dst) and
// the token sums (rows of ssrc by dest, into sdst).  CG = 2 launches clusters
// of two (as many pairs as are resident at once, fewer under a grid cap).
template <int KA, int KB, int NST, int CG>
int mega_launch(const moe_cfg& c, const WsLayout& L, uint8_t* ws, const GemmArgs& a, const uint16_t* gsrc,
                uint16_t* gdst, const float* ssrc, float* sdst, int grid, int trace_kind, cudaStream_t s) {
  MegaParams mp;
  std::memset(&mp, 0, sizeof(mp));
  if (!fill_params<KA, CG>(a, mp.g1) || !fill_params<KB, CG>(a, mp.g2)) return MOE_ERR_CUDA;
  // the whole ring, one CTA per SM (the grouped GEMMs' stage-count and
  // epilogue knobs do not apply here)
  mp.g1.nst = mp.g2.nst = NST;
  const long long R = static_cast<long long>(c.T) * c.k;
  // a gathered row must fit a ring stage
  if (2ll * c.d_model > Mega<KA, KB, NST, CG>::STAGE_BYTES) return MOE_ERR_SHAPE;
  mp.x = gsrc;
  mp.row_token = reinterpret_cast<const int32_t*>(ws + L.row_token);
  mp.dest = reinterpret_cast<const int32_t*>(ws + L.dest);
  mp.Xp = gdst;
  mp.Op = ssrc;
  mp.y = sdst;
  mp.ctr = reinterpret_cast<int*>(ws + L.mk);
  // 128-row gather tasks when every SM gets a few; 32-row ones for small
  // layers, whose gather would otherwise sit on a handful of CTAs.
  mp.grows = R >= 256ll * num_sms() ? 128 : kMegaGatherRows;
  mp.NG = ceil_div(R, mp.grows);
  mp.skip = g_skip_ticket;
  mp.trace = g_trace_buf;
  mp.trace_per_cta = g_trace_per_cta;
  // counters: kCtrXp + NG gather flags + (at most R/128 + E + S*ceil(T/128)) m-tiles
  const long long need = kCtrXp + mp.NG + R / kBM + c.E + static_cast<long long>(c.n_shared) * ceil_div(c.T, kBM) + 2;
  if (need > L.mk_ints) return MOE_ERR_SHAPE;
  if (cudaMemsetAsync(mp.ctr, 0, sizeof(int) * L.mk_ints, s) != cudaSuccess) return MOE_ERR_CUDA;
  constexpr int kSmem = mega_smem_bytes<KA, KB, NST, CG>();
  auto kern = mega_kernel<KA, KB, NST, CG>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return MOE_ERR_CUDA;
  int nblocks = grid > 0 ? grid : num_sms();
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  if constexpr (CG == 2) {
    const int cap = mega_pair_capacity<KA, KB, NST>();
    if (cap <= 0) return MOE_ERR_CUDA;
    nblocks = 2 * std::max(1, std::min(cap, nblocks / 2));
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cfg.gridDim = dim3(nblocks);
  TraceScope trace_scope(trace_kind, s);
  if (cudaLaunchKernelEx(&cfg, kern, mp) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// CTA pairs when both of the MegaKernel's GEMM kinds run on pairs as
// stand-alone kernels (moe_set_gemm_pair_kinds) and pairs can be resident.
template <int KA, int KB, int NST2>
bool mega_uses_pairs(int d) {
  const int mask = gemm_pair_kinds();
  return ((mask >> KA) & 1) && ((mask >> KB) & 1) && 2 * d <= Mega<KA, KB, NST2, 2>::STAGE_BYTES &&
         mega_pair_capacity<KA, KB, NST2>() > 0;
}

}  // namespace

int megakernel_fwd(const moe_cfg& c, const WsLayout& L, uint8_t* ws, const uint16_t* x, const uint16_t* W1,
                   const uint16_t* W3, const uint16_t* W2, const float* topk_w, float* y, int grid, cudaStream_t s) {
  GemmArgs a{};
  a.T = c.T;
  a.d = c.d_model;
  a.f = c.d_ff;
  a.E = c.E;
  a.k = c.k;
  a.S = c.n_shared;
  a.offsets = reinterpret_cast<const int32_t*>(ws + L.offsets);
  a.row_slot = reinterpret_cast<const int32_t*>(ws + L.row_slot);
  a.topk_w = topk_w;
  a.Xp = reinterpret_cast<const uint16_t*>(ws + L.Xp);
  a.x = x;
  a.W1 = W1;
  a.W3 = W3;
  a.W2 = W2;
  a.Hw = reinterpret_cast<const uint16_t*>(ws + L.Hw);
  a.Hw_out = reinterpret_cast<uint16_t*>(ws + L.Hw);
  a.AB_out = reinterpret_cast<uint16_t*>(ws + L.AB);
  a.Op_out = reinterpret_cast<float*>(ws + L.Op);
  a.err = reinterpret_cast<int*>(ws + L.err);
  uint16_t* Xp = reinterpret_cast<uint16_t*>(ws + L.Xp);
  const float* Op = reinterpret_cast<const float*>(ws + L.Op);
  if (mega_uses_pairs<kG1, kG2, 6>(c.d_model))
    return mega_launch<kG1, kG2, 6, 2>(c, L, ws, a, x, Xp, Op, y, grid, MOE_K_MEGAKERNEL, s);
  return mega_launch<kG1, kG2, 4, 1>(c, L, ws, a, x, Xp, Op, y, grid, MOE_K_MEGAKERNEL, s);
}

int megakernel_bwd_input(const moe_cfg& c, const WsLayout& L, uint8_t* ws, const GemmArgs& a, const uint16_t* dy,
                         float* dx, int grid, cudaStream_t s) {
  uint16_t* G = reinterpret_cast<uint16_t*>(ws + L.G);
  const float* dXp = reinterpret_cast<const float*>(ws + L.dXp);
  if (mega_uses_pairs<kDH, kDX, 6>(c.d_model))
    return mega_launch<kDH, kDX, 6, 2>(c, L, ws, a, dy, G, dXp, dx, grid, MOE_K_MEGAKERNEL_BWD, s);
  return mega_launch<kDH, kDX, 4, 1>(c, L, ws, a, dy, G, dXp, dx, grid, MOE_K_MEGAKERNEL_BWD, s);
}

}  // namespace moe

extern "C" int moe_debug_skip_megakernel_task(int ticket) {
  moe::g_skip_ticket = ticket >= 0 ? ticket : -1;
  return MOE_OK;
}

extern "C" int moe_debug_megakernel_trace(void* buf, int records_per_cta) {
  if (buf && (records_per_cta < 2 || (reinterpret_cast<uintptr_t>(buf) & 15u))) return MOE_ERR_ARG;
  moe::g_trace_buf = static_cast<unsigned long long*>(buf);
  moe::g_trace_per_cta = buf ? records_per_cta : 0;
  return MOE_OK;
}

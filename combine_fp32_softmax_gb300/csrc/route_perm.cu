// Router, deterministic token mapping, row gather and fixed-order row sums.
//
// Router: UniEP page ("Unified Expert-Parallel MoE MegaKernel for LLM
// Training"), section 1.1: the gating network gives each token a probability
// per expert, then top-k picks the target experts.
// Token mapping: same page, section 2.2, Algorithm 1 (deterministic global
// token mapping): a local stable sort by expert plus prefix-sum base offsets
// gives every (token, slot) a unique, conflict-free address without atomics
// on the addresses; with one rank the cross-rank base is 0.  Here the
// "stable sort" is a per-block expert histogram, one flat exclusive scan over
// the expert-major [E][blocks] table, and an in-block stable rank from warp
// match/ballot masks.
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "trace.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;
// One warp per token: a token's softmax and top-k are a serial chain of
// shuffles, so the parallelism is in the tokens (a block is the 32 tokens of
// one histogram block).
constexpr int kRouteWarps = kRouteTokensPerBlock;
constexpr int kMaxRowsPerToken = 12;  // k <= 8 routed + S <= 4 shared

// Softmax statistics of one logit row held lane-strided by a warp
// (expert e = lane + 32 * i).  Router forward and backward both use this,
// so the backward's probabilities are bit-identical to the forward's.
template <int EPL>
struct RowSoftmax {
  float v[EPL];   // logits (-inf beyond E)
  float ex[EPL];  // expf(v - m) (0 beyond E)
  float m, s;     // max, sum of ex
};

// One logit row, lane-strided (-inf beyond E).
template <int EPL>
__device__ __forceinline__ void row_load(const float* __restrict__ row, int E, int lane, float (&v)[EPL]) {
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? row[e] : -INFINITY;
  }
}

// Order-preserving key of a finite float: a larger value has a larger
// unsigned key, -0.0 and +0.0 share one, and every finite value's key is
// above 0 (the key of "no entry").  Warp max/min over keys are single
// redux.sync instructions, where a float max needs a shuffle butterfly.
__device__ __forceinline__ unsigned order_key(float v) {
  const unsigned u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Softmax statistics of the row already in r.v; false if it holds a
// non-finite logit (the statistics are then unspecified).  key[i] is the
// order key of entry i (0 beyond E).
template <int EPL>
__device__ __forceinline__ bool row_stats(int E, int lane, RowSoftmax<EPL>& r, unsigned (&key)[EPL]) {
  bool bad = false;
  unsigned kmax = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E && !isfinite(r.v[i])) bad = true;
    key[i] = e < E ? order_key(r.v[i]) : 0u;
    kmax = max(kmax, key[i]);
  }
  bad = __any_sync(kFull, bad);
  // The maximum is exact whichever way it is found; -0.0 and +0.0 give the
  // same exp(v - m) bits.
  const float m = key_value(__reduce_max_sync(kFull, kmax));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    r.ex[i] = (e < E) ? expf(r.v[i] - m) : 0.f;
    s += r.ex[i];
  }
  // xor butterfly: every lane adds the same pairs, so all lanes end with
  // the same bits.
#pragma unroll
  for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
  r.m = m;
  r.s = s;
  return !bad;
}

template <int EPL>
__device__ __forceinline__ bool row_softmax(const float* __restrict__ row, int E, int lane, RowSoftmax<EPL>& r) {
  row_load<EPL>(row, E, lane, r.v);
  unsigned key[EPL];
  return row_stats<EPL>(E, lane, r, key);
}

// Routes token t on one warp (its logit row already in r.v): softmax
// statistics, then k rounds of warp argmax.  Lane j < k ends with slot j's
// expert and weight.  A row with a non-finite logit is reported and gets the
// placeholder routing slot j -> expert j with weight 0.
template <int EPL>
__device__ __forceinline__ void route_token(RowSoftmax<EPL>& r, int t, int E, int k, int renorm, int lane, int* err,
                                            int& my_idx, float& my_w) {
  my_idx = lane;
  my_w = 0.f;
  unsigned key[EPL];
  if (!row_stats<EPL>(E, lane, r, key)) {
    if (lane == 0) record_error(err, MOE_ERR_NONFINITE_CODE, t);
    return;
  }
  float psum = 0.f, my_p = 0.f;
  for (int j = 0; j < k; ++j) {
    // Best remaining entry of this lane: strictly greater keeps the lower
    // index on ties (entries are visited in increasing expert index).
    unsigned bk = 0;
    unsigned be = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (key[i] > bk) {
        bk = key[i];
        be = static_cast<unsigned>(lane + 32 * i);
      }
    // Winner under (value desc, index asc), a strict total order: the
    // largest key, then the lowest expert index holding it.  Every lane
    // gets the same winner.
    const unsigned kbest = __reduce_max_sync(kFull, bk);
    const int bi = static_cast<int>(__reduce_min_sync(kFull, bk == kbest ? be : 0xffffffffu));
    const int owner = bi & 31, which = bi >> 5;
    float p_local = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane == owner && i == which) {
        key[i] = 0u;  // taken
        p_local = r.ex[i] / r.s;
      }
    const float p = __shfl_sync(kFull, p_local, owner);
    if (lane == j) {
      my_idx = bi;
      my_p = p;
    }
    psum += p;
  }
  my_w = renorm ? my_p / psum : my_p;
}

// Routes the 32 tokens of histogram block hb (warp w: token 32*hb + w) and
// counts their slots per expert in s_hist (zeroed by the caller).
template <int EPL>
__device__ __forceinline__ void route_block(const float* __restrict__ logits, int hb, int T, int E, int k, int renorm,
                                            int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int* s_hist,
                                            int* err) {
  static_assert(kRouteWarps == kRouteTokensPerBlock, "one warp per token");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = hb * kRouteTokensPerBlock + warp;
  if (t >= T) return;
  RowSoftmax<EPL> r;
  row_load<EPL>(logits + static_cast<size_t>(t) * E, E, lane, r.v);
  int my_idx;
  float my_w;
  route_token<EPL>(r, t, E, k, renorm, lane, err, my_idx, my_w);
  if (lane < k) {
    topk_idx[static_cast<size_t>(t) * k + lane] = my_idx;
    topk_w[static_cast<size_t>(t) * k + lane] = my_w;
    atomicAdd(&s_hist[my_idx], 1);  // integer count: order-independent
  }
}

template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
    route_kernel(const float* __restrict__ logits, int T, int E, int k, int renorm, int32_t* __restrict__ topk_idx,
                 float* __restrict__ topk_w, int32_t* __restrict__ hist, int nb, int* err) {
  __shared__ int s_hist[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  route_block<EPL>(logits, blockIdx.x, T, E, k, renorm, topk_idx, topk_w, s_hist, err);
  __syncthreads();
  if (hist)
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<size_t>(e) * nb + blockIdx.x] = s_hist[e];
}

// Histogram of caller-provided expert indices (moe_dispatch without the
// router).  Out-of-range indices are clamped (and reported) so the tables
// stay a valid permutation.
__global__ void __launch_bounds__(256)
    hist_kernel(const int32_t* __restrict__ topk_idx, int T, int E, int k, int32_t* __restrict__ hist, int nb,
                int* err) {
  __shared__ int s_hist[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  const size_t s0 = static_cast<size_t>(blockIdx.x) * kRouteTokensPerBlock * k;
  const int nslot = (min(T, (blockIdx.x + 1) * kRouteTokensPerBlock) - blockIdx.x * kRouteTokensPerBlock) * k;
  for (int i = threadIdx.x; i < nslot; i += blockDim.x) {
    int e = topk_idx[s0 + i];
    if (e < 0 || e >= E) {
      record_error(err, MOE_ERR_ARG, static_cast<int>(s0 + i));
      e = min(max(e, 0), E - 1);
    }
    atomicAdd(&s_hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<size_t>(e) * nb + blockIdx.x] = s_hist[e];
}

// Exclusive scan of in[0, n) into out by one kScanThreads-thread block;
// returns the total to every thread.  The array is scanned in tiles of
// kScanTile entries: each tile is loaded coalesced into shared memory (entry
// i at i + i/32, so a warp reading 8 consecutive entries per thread hits
// every bank once), each thread sums its 8 entries, a two-level warp shuffle
// scan gives every thread its exclusive prefix, and the prefixes go back out
// coalesced; a carry runs across tiles.  in is read through L2 only (it may
// have been written by other blocks of the same launch).
constexpr int kScanThreads = 1024;
constexpr int kScanPer = 8;
constexpr int kScanTile = kScanThreads * kScanPer;

struct ScanSmem {
  int tile[kScanTile + kScanTile / 32];
  int warp_tot[32];
  int tile_total;
};

__device__ __forceinline__ int block_exclusive_scan(const int32_t* in, int n, int32_t* out, ScanSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int carry = 0;
  for (int t0 = 0; t0 < n; t0 += kScanTile) {
    const int m = min(kScanTile, n - t0);
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) {
      const int i = tid + j * kScanThreads;
      sm.tile[i + (i >> 5)] = i < m ? __ldcg(in + t0 + i) : 0;
    }
    __syncthreads();
    int v[kScanPer];
    int local = 0;
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) {
      const int i = tid * kScanPer + j;
      v[j] = sm.tile[i + (i >> 5)];
      local += v[j];
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) sm.warp_tot[w] = incl;
    __syncthreads();
    if (w == 0) {
      const int x = sm.warp_tot[lane];
      int inc = x;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(kFull, inc, off);
        if (lane >= off) inc += y;
      }
      sm.warp_tot[lane] = inc - x;
      if (lane == 31) sm.tile_total = inc;
    }
    __syncthreads();
    int run = carry + sm.warp_tot[w] + incl - local;
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) {
      const int i = tid * kScanPer + j;
      sm.tile[i + (i >> 5)] = run;
      run += v[j];
    }
    carry += sm.tile_total;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) {
      const int i = tid + j * kScanThreads;
      if (i < m) out[t0 + i] = sm.tile[i + (i >> 5)];
    }
    __syncthreads();  // tile, warp_tot and tile_total are rewritten by the next tile
  }
  return carry;
}

// One flat exclusive scan of the expert-major [E][nb] histogram: at (e, b)
// it equals offsets[e] + (slots of expert e in blocks < b), i.e. the base
// address of block b's first slot for expert e.
__global__ void __launch_bounds__(kScanThreads)
    scan_kernel(const int32_t* __restrict__ hist, int E, int nb, int R, int32_t* __restrict__ base,
                int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  __shared__ ScanSmem sm;
  block_exclusive_scan(hist, E * nb, base, sm);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int b0 = base[static_cast<size_t>(e) * nb];
    const int b1 = (e + 1 < E) ? base[static_cast<size_t>(e + 1) * nb] : R;
    offsets[e] = b0;
    counts[e] = b1 - b0;
  }
  if (threadIdx.x == 0) offsets[E] = R;
}

// Stable in-block ranks of histogram block hb on NW warps.  Warp w owns
// tokens [TPW*w, TPW*w+TPW) of the block, i.e. a contiguous run of TPW*k flat
// slots, visited in rounds of 32.  Pass 1 counts per (warp, expert); a prefix
// over warps (starting at the block's global base for the expert, plus
// off[e] where the base holds only the within-expert prefix) gives each
// warp's first address per expert; pass 2 ranks each slot among
// equal-expert lanes of its round (match mask) and advances.  The result
// does not depend on NW: a slot's address is its expert's base plus the
// number of earlier slots of the block with the same expert.
template <int NW>
__device__ __forceinline__ void scatter_block(const int32_t* __restrict__ topk_idx, const int32_t* base,
                                              const int* off, int hb, int T, int E, int k, int nb,
                                              int (*wrun)[256], int32_t* __restrict__ dest,
                                              int32_t* __restrict__ row_token, int32_t* __restrict__ row_slot,
                                              int* err) {
  constexpr int TPW = kRouteTokensPerBlock / NW;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int i = tid; i < NW * 256; i += NW * 32) (&wrun[0][0])[i] = 0;
  __syncthreads();
  const size_t slot0 = static_cast<size_t>(hb) * kRouteTokensPerBlock * k;
  const int nslot = (min(T, (hb + 1) * kRouteTokensPerBlock) - hb * kRouteTokensPerBlock) * k;
  const int wslots = TPW * k;
  const int wslot0 = w * wslots;
  const int rounds = (wslots + 31) / 32;
  for (int rnd = 0; rnd < rounds; ++rnd) {
    const int il = wslot0 + rnd * 32 + lane;
    const bool valid = rnd * 32 + lane < wslots && il < nslot;
    const int e = valid ? min(max(__ldcg(topk_idx + slot0 + il), 0), E - 1) : -1;
    const unsigned peers = __match_any_sync(kFull, e);
    if (valid && lane == __ffs(peers) - 1) wrun[w][e] += __popc(peers);
  }
  __syncthreads();
  for (int e = tid; e < E; e += NW * 32) {
    int run = __ldcg(base + static_cast<size_t>(e) * nb + hb) + (off ? off[e] : 0);
#pragma unroll
    for (int ww = 0; ww < NW; ++ww) {
      const int c = wrun[ww][e];
      wrun[ww][e] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int rnd = 0; rnd < rounds; ++rnd) {
    const int il = wslot0 + rnd * 32 + lane;
    const bool valid = rnd * 32 + lane < wslots && il < nslot;
    const int e = valid ? min(max(__ldcg(topk_idx + slot0 + il), 0), E - 1) : -1;
    const unsigned peers = __match_any_sync(kFull, e);
    const int r = valid ? wrun[w][e] + __popc(peers & lt) : 0;
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) wrun[w][e] += __popc(peers);
    __syncwarp();
    if (valid && (row_token == nullptr ||
                  debug_ok(static_cast<unsigned>(r) < static_cast<unsigned>(T * k), err, kDbgPermRow, slot0 + il))) {
      const size_t i = slot0 + il;
      dest[i] = r;
      if (row_token) {  // inverse tables only when the addresses are local rows
        row_token[r] = static_cast<int>(i / k);
        row_slot[r] = static_cast<int>(i);
      }
    }
  }
}

constexpr int kScatterWarps = 8;

__global__ void __launch_bounds__(kScatterWarps * 32)
    scatter_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ base, int T, int E, int k,
                   int nb, int32_t* __restrict__ dest, int32_t* __restrict__ row_token,
                   int32_t* __restrict__ row_slot, int* err) {
  __shared__ int wrun[kScatterWarps][256];
  scatter_block<kScatterWarps>(topk_idx, base, nullptr, blockIdx.x, T, E, k, nb, wrun, dest, row_token, row_slot,
                               err);
}

// Grid barrier of a cooperative launch (every block resident at once).
// Thread 0 of each block reads the generation, publishes the block's writes
// and arrives; the last arrival resets the count and advances the
// generation; the others spin on the generation for at most kWaitLimitNs.
// On a timeout (recorded in err) it returns false in every thread of the
// block; the count is then left inconsistent until moe_ws_init.
__device__ bool grid_barrier(int* bar, int* err, int where) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const int gen = ld_acquire_gpu(bar + 1);
    __threadfence();
    if (atomicAdd(bar, 1) == static_cast<int>(gridDim.x) - 1) {
      __threadfence();
      atomicExch(bar, 0);
      red_release_gpu_add(bar + 1, 1);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(bar + 1) == gen) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          record_error(err, MOE_ERR_TIMEOUT_CODE, where);
          ok = 0;
          break;
        }
        __nanosleep(32);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// After a timed-out grid barrier: placeholder tables that keep the later
// kernels of the call in bounds (every slot to its own row, all rows in the
// last expert); the error word already marks the results void.  Blocks that
// passed the barrier write the real tables, which are in range as well.
__device__ void placeholder_tables(int T, int E, int k, int nb, int32_t* counts, int32_t* offsets, int32_t* dest,
                                   int32_t* row_token, int32_t* row_slot) {
  const int R = T * k;
  for (int hb = blockIdx.x; hb < nb; hb += gridDim.x) {
    const int i0 = hb * kRouteTokensPerBlock * k, i1 = min(R, i0 + kRouteTokensPerBlock * k);
    for (int i = i0 + static_cast<int>(threadIdx.x); i < i1; i += blockDim.x) {
      dest[i] = i;
      row_token[i] = i / k;
      row_slot[i] = i;
    }
  }
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      offsets[e] = 0;
      counts[e] = e == E - 1 ? R : 0;
    }
    if (threadIdx.x == 0) offsets[E] = R;
  }
}

// Scratch of the fused kernel, one phase at a time.
union RouteTablesSmem {
  int hist[256];
  ScanSmem scan;
  struct {
    int wrun[kRouteWarps][256];
    int off[256];
  } scatter;
};

// Router and permutation builder in one cooperative launch: the same three
// steps as route_kernel, scan_kernel and scatter_kernel, with grid barriers
// in place of kernel boundaries, so the tables are bit-identical to theirs.
//   1. Each block routes histogram blocks hb = blockIdx.x, + gridDim.x, ...
//      and writes their expert counts hist[e][hb].
//   2. Each block scans whole expert rows: base[e][b] = slots of expert e
//      in blocks < b, counts[e] = the row's total.
//   3. Every block turns counts into offsets (block 0 stores them) and
//      ranks its histogram blocks' slots (address = offsets[e] + base[e][b]
//      + earlier slots of block b with expert e).
// Two CTAs per SM (32 registers a thread) where the router's rows fit.
template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32, EPL <= 4 ? 2 : 1)
    route_tables_kernel(const float* __restrict__ logits, int T, int E, int k, int renorm, int nb, int R,
                        int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ hist,
                        int32_t* __restrict__ base, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                        int32_t* __restrict__ dest, int32_t* __restrict__ row_token,
                        int32_t* __restrict__ row_slot, int* err) {
  __shared__ RouteTablesSmem sm;
  griddep_launch_dependents();
  int* bar = err + kErrBarrierWord;
  for (int hb = blockIdx.x; hb < nb; hb += gridDim.x) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) sm.hist[e] = 0;
    __syncthreads();
    route_block<EPL>(logits, hb, T, E, k, renorm, topk_idx, topk_w, sm.hist, err);
    __syncthreads();
    // Thread e reads sm.hist[e] here and zeroes it next iteration itself.
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<size_t>(e) * nb + hb] = sm.hist[e];
  }
  if (!grid_barrier(bar, err, 1)) {
    placeholder_tables(T, E, k, nb, counts, offsets, dest, row_token, row_slot);
    return;
  }
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const size_t row = static_cast<size_t>(e) * nb;
    const int total = block_exclusive_scan(hist + row, nb, base + row, sm.scan);
    if (threadIdx.x == 0) counts[e] = total;
  }
  if (!grid_barrier(bar, err, 2)) {
    placeholder_tables(T, E, k, nb, counts, offsets, dest, row_token, row_slot);
    return;
  }
  if (threadIdx.x < 32) {  // E <= 256: eight experts per lane
    const int lane = threadIdx.x;
    int v[8];
    int local = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      v[j] = e < E ? __ldcg(counts + e) : 0;
      local += v[j];
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += y;
    }
    int run = incl - local;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      if (e < E) {
        sm.scatter.off[e] = run;
        if (blockIdx.x == 0) offsets[e] = run;
      }
      run += v[j];
    }
    if (blockIdx.x == 0 && lane == 0) offsets[E] = R;
  }
  __syncthreads();
  for (int hb = blockIdx.x; hb < nb; hb += gridDim.x) {
    scatter_block<kRouteWarps>(topk_idx, base, sm.scatter.off, hb, T, E, k, nb, sm.scatter.wrun, dest, row_token,
                               row_slot, err);
    __syncthreads();  // the next block zeroes wrun
  }
}

// Cross-rank bases of the multi-rank token mapping (one block of 256
// threads, thread e = expert e).  counts is the all-gathered [G][E] table of
// every rank's per-expert slot counts.  Expert e's segment starts, inside
// its owner's receive buffer, after the segments of the lower experts with
// the same owner; within it rank r's slots follow those of ranks < r.  All
// sums run in a fixed (ascending) order.
__global__ void __launch_bounds__(256)
    rank_bases_kernel(const int32_t* __restrict__ counts, int G, int E, const int32_t* __restrict__ owner, int rank,
                      int32_t* __restrict__ rank_base, int32_t* __restrict__ recv_rows) {
  __shared__ int s_total[256], s_owner[256];
  const int e = threadIdx.x;
  int lower = 0;
  if (e < E) {
    int total = 0;
    for (int g = 0; g < G; ++g) {
      const int c = counts[static_cast<size_t>(g) * E + e];
      if (g < rank) lower += c;
      total += c;
    }
    s_total[e] = total;
    s_owner[e] = min(max(owner[e], 0), G - 1);
  }
  __syncthreads();
  if (e < E) {
    int start = 0;
    for (int u = 0; u < e; ++u)
      if (s_owner[u] == s_owner[e]) start += s_total[u];
    rank_base[e] = start + lower;
  }
  if (recv_rows)
    for (int o = threadIdx.x; o < G; o += blockDim.x) {
      int rows = 0;
      for (int u = 0; u < E; ++u)
        if (s_owner[u] == o) rows += s_total[u];
      recv_rows[o] = rows;
    }
}

// Moves every block base of expert e from the local segment start
// offsets[e] to the rank's global base rank_base[e] (multi-rank mapping).
__global__ void rebase_kernel(int32_t* __restrict__ base, const int32_t* __restrict__ offsets,
                              const int32_t* __restrict__ rank_base, int E, int nb) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= E * nb) return;
  const int e = i / nb;
  base[i] += rank_base[e] - offsets[e];
}

// dst[r] = src[idx[r]]: one warp per row, 16-byte vectors, kGatherVec in
// flight per lane (a whole 4 KB row of d = 2048 bf16); the next row's index
// is loaded before the current row is copied.  An index outside [0, nsrc)
// writes a zero row.
constexpr int kGatherVec = 8;

__global__ void __launch_bounds__(256)
    gather_rows_bf16_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ idx, int nsrc, int nrows,
                            int nvec, uint4* __restrict__ dst, int* err) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int sr = r < nrows ? idx[r] : 0;
  for (; r < nrows; r += nwarps) {
    const int rn = r + nwarps;
    const int sr_next = rn < nrows ? idx[rn] : 0;
    const bool ok = static_cast<unsigned>(sr) < static_cast<unsigned>(nsrc);
    if (lane == 0) debug_ok(ok, err, kDbgGatherRow, r);
    const uint4* s = src + static_cast<size_t>(ok ? sr : 0) * nvec;
    uint4* o = dst + static_cast<size_t>(r) * nvec;
    for (int v = lane; v < nvec; v += 32 * kGatherVec) {
      uint4 t[kGatherVec];
#pragma unroll
      for (int u = 0; u < kGatherVec; ++u)
        if (v + 32 * u < nvec) t[u] = ok ? __ldg(s + v + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < kGatherVec; ++u)
        if (v + 32 * u < nvec) o[v + 32 * u] = t[u];
    }
    sr = sr_next;
  }
}

// dst[dest[t*k + j]] = src[t] for every token t and slot j < k: the same
// rows a gather by row_token writes, but each source row is read once and
// written k times, so a source larger than L2 is streamed from HBM once
// instead of k times.  A warp's unit is one token's span of 32*kGatherVec
// vectors (kGatherVec in flight per lane); the grid is the resident
// capacity.  A destination outside [0, ndst) is skipped.
__global__ void __launch_bounds__(256)
    scatter_rows_bf16_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ dest, int T, int k,
                             int ndst, int nvec, uint4* __restrict__ dst, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int kSpan = 32 * kGatherVec;
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int spans = (nvec + kSpan - 1) / kSpan;
  const int units = T * spans;  // < 2^31: checked by the launcher
  for (int u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += nwarps) {
    const int t = u / spans;
    const int v0 = (u - t * spans) * kSpan + lane;
    const int mydest = lane < k ? dest[static_cast<size_t>(t) * k + lane] : -1;
    const uint4* s = src + static_cast<size_t>(t) * nvec;
    uint4 val[kGatherVec];
#pragma unroll
    for (int i = 0; i < kGatherVec; ++i)
      if (v0 + 32 * i < nvec) val[i] = __ldg(s + v0 + 32 * i);
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(kFull, mydest, j);
      if (lane == 0 && v0 == 0) debug_ok(static_cast<unsigned>(r) < static_cast<unsigned>(ndst), err, kDbgScatterRow, t);
      if (static_cast<unsigned>(r) >= static_cast<unsigned>(ndst)) continue;
      uint4* o = dst + static_cast<size_t>(r) * nvec;
#pragma unroll
      for (int i = 0; i < kGatherVec; ++i)
        if (v0 + 32 * i < nvec) o[v0 + 32 * i] = val[i];
    }
  }
}

// out[t] = ((rows[sel[t*k]] + rows[sel[t*k+1]]) + ...) + rows[R + t] + ...
// in exactly that order, fp32, one warp per token.  NR = k + S rows per
// token is a template parameter so the loads of every row (two float4 per
// lane per step) are in registers with no spare slots, which keeps enough
// warps resident to stream at HBM rate.
// A warp's unit of work is one token's span of kSumSpan float4 columns, so
// the work divides into many more units than there are resident warps and
// the last wave is short; the grid is the resident capacity.
constexpr int kSumSpan = 128;

template <int NR>
__global__ void __launch_bounds__(256)
    sum_rows_f32_kernel(const float4* __restrict__ rows, const int32_t* __restrict__ sel, int T, int k, int S,
                        int nvec, float4* __restrict__ out, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const long long R = static_cast<long long>(T) * k;
  const long long nrows = R + static_cast<long long>(S) * T;
  const int spans = (nvec + kSumSpan - 1) / kSumSpan;
  const int units = T * spans;  // < 2^31: checked by the launcher
  for (int u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += nwarps) {
    const int t = u / spans;
    const int v0 = (u - t * spans) * kSumSpan;
    const int v1 = min(nvec, v0 + kSumSpan);
    long long myrow = 0;
    if (lane < k) {
      myrow = sel[static_cast<size_t>(t) * k + lane];
      if (v0 == 0) debug_ok(myrow >= 0 && myrow < nrows, err, kDbgSumRow, t);
      if (myrow < 0 || myrow >= nrows) myrow = 0;
    } else if (lane < NR) {
      myrow = R + static_cast<long long>(lane - k) * T + t;
    }
    const float4* base[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) base[j] = rows + static_cast<size_t>(__shfl_sync(kFull, myrow, j)) * nvec;
    float4* o = out + static_cast<size_t>(t) * nvec;
    for (int v = v0 + lane; v < v1; v += 64) {
      const bool two = v + 32 < v1;
      float4 val[NR], val2[NR];
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        val[j] = __ldg(base[j] + v);
        val2[j] = two ? __ldg(base[j] + v + 32) : val[j];
      }
      float4 acc = val[0], acc2 = val2[0];
#pragma unroll
      for (int j = 1; j < NR; ++j) {
        acc.x += val[j].x;
        acc.y += val[j].y;
        acc.z += val[j].z;
        acc.w += val[j].w;
        acc2.x += val2[j].x;
        acc2.y += val2[j].y;
        acc2.z += val2[j].z;
        acc2.w += val2[j].w;
      }
      o[v] = acc;
      if (two) o[v + 32] = acc2;
    }
  }
}

// dw[i] = sum over column tiles n (in order) of partial[dest[i] * nt + n].
__global__ void dw_reduce_kernel(const float* __restrict__ partial, const int32_t* __restrict__ dest, int R, int nt,
                                 float* __restrict__ dw, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= R) return;
  if (!debug_ok(static_cast<unsigned>(dest[i]) < static_cast<unsigned>(R), err, kDbgDwReduce, i)) return;
  const size_t r = static_cast<size_t>(dest[i]);
  float s = 0.f;
  for (int n = 0; n < nt; ++n) s += partial[r * nt + n];
  dw[i] = s;
}

// Router backward (softmax Jacobian restricted to the picked experts'
// weights), one warp per token.
template <int EPL>
__global__ void __launch_bounds__(256)
    route_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                     const float* __restrict__ topk_w, const float* __restrict__ dw, int T, int E, int k, int renorm,
                     float* __restrict__ dlogits, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nwarps) {
    RowSoftmax<EPL> r;
    const bool ok = row_softmax<EPL>(logits + static_cast<size_t>(t) * E, E, lane, r);
    int my_idx = -1;
    float my_w = 0.f, my_dw = 0.f;
    if (lane < k) {
      my_idx = topk_idx[static_cast<size_t>(t) * k + lane];
      debug_ok(static_cast<unsigned>(my_idx) < static_cast<unsigned>(E), err, kDbgRouteBwd, t);
      my_w = topk_w[static_cast<size_t>(t) * k + lane];
      my_dw = dw[static_cast<size_t>(t) * k + lane];
    }
    // One pass over the k slots: inner = sum_j dw_j w_j in slot order, and
    // each entry this lane holds learns whether (and in which slot) it was
    // picked.
    float inner = 0.f;
    float pick_dw[EPL], pick_w[EPL];
    bool picked[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      pick_dw[i] = pick_w[i] = 0.f;
      picked[i] = false;
    }
    for (int j = 0; j < k; ++j) {
      const int sj = __shfl_sync(kFull, my_idx, j);
      const float dj = __shfl_sync(kFull, my_dw, j);
      const float wj = __shfl_sync(kFull, my_w, j);
      inner += dj * wj;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (sj == lane + 32 * i) {
          picked[i] = true;
          pick_dw[i] = dj;
          pick_w[i] = wj;
        }
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        float dz;
        if (!ok)
          dz = 0.f;
        else if (renorm == 0)
          dz = (r.ex[i] / r.s) * ((picked[i] ? pick_dw[i] : 0.f) - inner);
        else
          dz = picked[i] ? pick_w[i] * (pick_dw[i] - inner) : 0.f;
        dlogits[static_cast<size_t>(t) * E + e] = dz;
      }
    }
  }
}

int sm_count_cached() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

}  // namespace

int num_sms() { return sm_count_cached(); }

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* topk_idx, float* topk_w,
                         int32_t* hist, int nb, int* err, cudaStream_t s) {
  TraceScope trace_scope(MOE_K_ROUTE, s);
  const dim3 grid(ceil_div(T, kRouteTokensPerBlock)), block(kRouteWarps * 32);
  if (E <= 32)
    route_kernel<1><<<grid, block, 0, s>>>(logits, T, E, k, renorm, topk_idx, topk_w, hist, nb, err);
  else if (E <= 64)
    route_kernel<2><<<grid, block, 0, s>>>(logits, T, E, k, renorm, topk_idx, topk_w, hist, nb, err);
  else if (E <= 128)
    route_kernel<4><<<grid, block, 0, s>>>(logits, T, E, k, renorm, topk_idx, topk_w, hist, nb, err);
  else
    route_kernel<8><<<grid, block, 0, s>>>(logits, T, E, k, renorm, topk_idx, topk_w, hist, nb, err);
  return cudaGetLastError();
}

namespace {
template <int EPL>
cudaError_t launch_route_tables_epl(const float* logits, int T, int E, int k, int renorm, int nb, int32_t* topk_idx,
                                    float* topk_w, int32_t* hist, int32_t* base, int32_t* counts, int32_t* offsets,
                                    int32_t* dest, int32_t* row_token, int32_t* row_slot, int* err, int max_grid,
                                    cudaStream_t s) {
  static int per_sm = 0;  // blocks of this kernel resident per SM
  if (per_sm == 0) {
    int n = 0;
    const cudaError_t e =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, route_tables_kernel<EPL>, kRouteWarps * 32, 0);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorCooperativeLaunchTooLarge;
    per_sm = n;
  }
  int grid = std::min(nb, per_sm * num_sms());
  if (max_grid > 0) grid = std::min(grid, max_grid);
  int R = T * k;
  void* args[] = {&logits, &T,    &E,      &k,    &renorm,    &nb,       &R,   &topk_idx, &topk_w,
                  &hist,   &base, &counts, &offsets, &dest, &row_token, &row_slot, &err};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(route_tables_kernel<EPL>), dim3(grid),
                                     dim3(kRouteWarps * 32), args, 0, s);
}
}  // namespace

cudaError_t launch_route_tables(const float* logits, int T, int E, int k, int renorm, int nb, int32_t* topk_idx,
                                float* topk_w, int32_t* hist, int32_t* base, int32_t* counts, int32_t* offsets,
                                int32_t* dest, int32_t* row_token, int32_t* row_slot, int* err, int max_grid,
                                cudaStream_t s) {
  TraceScope trace_scope(MOE_K_ROUTE_TABLES, s);
#define MOE_ROUTE_TABLES(EPL)                                                                                    \
  launch_route_tables_epl<EPL>(logits, T, E, k, renorm, nb, topk_idx, topk_w, hist, base, counts, offsets, dest, \
                               row_token, row_slot, err, max_grid, s)
  if (E <= 32) return MOE_ROUTE_TABLES(1);
  if (E <= 64) return MOE_ROUTE_TABLES(2);
  if (E <= 128) return MOE_ROUTE_TABLES(4);
  return MOE_ROUTE_TABLES(8);
#undef MOE_ROUTE_TABLES
}

cudaError_t launch_hist(const int32_t* topk_idx, int T, int E, int k, int32_t* hist, int nb, int* err,
                        cudaStream_t s) {
  TraceScope trace_scope(MOE_K_HIST, s);
  hist_kernel<<<nb, 256, 0, s>>>(topk_idx, T, E, k, hist, nb, err);
  return cudaGetLastError();
}

cudaError_t launch_scan(const int32_t* hist, int E, int nb, int R, int32_t* base, int32_t* counts, int32_t* offsets,
                        cudaStream_t s) {
  TraceScope trace_scope(MOE_K_SCAN, s);
  scan_kernel<<<1, 1024, 0, s>>>(hist, E, nb, R, base, counts, offsets);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const int32_t* topk_idx, const int32_t* base, int T, int E, int k, int nb, int32_t* dest,
                           int32_t* row_token, int32_t* row_slot, int* err, cudaStream_t s) {
  TraceScope trace_scope(MOE_K_SCATTER, s);
  scatter_kernel<<<nb, 256, 0, s>>>(topk_idx, base, T, E, k, nb, dest, row_token, row_slot, err);
  return cudaGetLastError();
}

cudaError_t launch_rebase(int32_t* base, const int32_t* offsets, const int32_t* rank_base, int E, int nb,
                          cudaStream_t s) {
  TraceScope trace_scope(MOE_K_SCAN, s);
  rebase_kernel<<<ceil_div(static_cast<long long>(E) * nb, 256), 256, 0, s>>>(base, offsets, rank_base, E, nb);
  return cudaGetLastError();
}

cudaError_t launch_rank_bases(const int32_t* counts, int G, int E, const int32_t* owner, int rank,
                              int32_t* rank_base, int32_t* recv_rows, cudaStream_t s) {
  TraceScope trace_scope(MOE_K_SCAN, s);
  rank_bases_kernel<<<1, 256, 0, s>>>(counts, G, E, owner, rank, rank_base, recv_rows);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows_bf16(const uint16_t* src, const int32_t* idx, int nsrc, int nrows, int d,
                                    uint16_t* dst, int trace_kind, int* err, cudaStream_t s) {
  if (nrows <= 0) return cudaSuccess;
  TraceScope trace_scope(trace_kind, s);
  static int resident = 0;  // blocks resident at once
  if (resident == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_rows_bf16_kernel, 256, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    resident = per_sm * num_sms();
  }
  const int blocks = min(ceil_div(nrows, 8), resident);
  gather_rows_bf16_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(src), idx, nsrc, nrows, d / 8,
                                                 reinterpret_cast<uint4*>(dst), err);
  return cudaGetLastError();
}

cudaError_t launch_scatter_rows_bf16(const uint16_t* src, const int32_t* dest, int T, int k, int d, uint16_t* dst,
                                     int trace_kind, int* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const long long units = static_cast<long long>(T) * ceil_div(d / 8, 32 * kGatherVec);
  if (units >= (1ll << 31) || static_cast<long long>(T) * k >= (1ll << 31)) return cudaErrorInvalidValue;
  TraceScope trace_scope(trace_kind, s);
  static int resident = 0;  // blocks resident at once
  if (resident == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, scatter_rows_bf16_kernel, 256, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    resident = per_sm * num_sms();
  }
  const int blocks = static_cast<int>(std::min<long long>(ceil_div(units, 8), resident));
  return launch_pdl(scatter_rows_bf16_kernel, dim3(blocks), dim3(256), 0, s, reinterpret_cast<const uint4*>(src),
                    dest, T, k, T * k, d / 8, reinterpret_cast<uint4*>(dst), err);
}

cudaError_t launch_sum_rows_f32(const float* rows, const int32_t* sel, int T, int k, int S, int d, float* out,
                                int trace_kind, int* err, cudaStream_t s) {
  TraceScope trace_scope(trace_kind, s);
  const long long units = static_cast<long long>(T) * ceil_div(d / 4, kSumSpan);
  if (units >= (1ll << 31)) return cudaErrorInvalidValue;
  const float4* r4 = reinterpret_cast<const float4*>(rows);
  float4* o4 = reinterpret_cast<float4*>(out);
  // Grid: the blocks that are resident at once (cached per row count), or
  // fewer when there is less work.
  auto grid_for = [&](auto kern, int nr) {
    static int resident[kMaxRowsPerToken + 1] = {0};
    if (resident[nr] == 0) {
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
      resident[nr] = per_sm * num_sms();
    }
    return static_cast<int>(std::min<long long>(ceil_div(units, 8), resident[nr]));
  };
  cudaError_t e = cudaSuccess;
  switch (k + S) {
#define MOE_SUM_ROWS_CASE(N) \
  case N:                                                                                           \
    e = launch_pdl(sum_rows_f32_kernel<N>, dim3(grid_for(sum_rows_f32_kernel<N>, N)), dim3(256), 0, s, r4, sel, T, k, \
                   S, d / 4, o4, err);                                                                                \
    break;
    MOE_SUM_ROWS_CASE(1)
    MOE_SUM_ROWS_CASE(2)
    MOE_SUM_ROWS_CASE(3)
    MOE_SUM_ROWS_CASE(4)
    MOE_SUM_ROWS_CASE(5)
    MOE_SUM_ROWS_CASE(6)
    MOE_SUM_ROWS_CASE(7)
    MOE_SUM_ROWS_CASE(8)
    MOE_SUM_ROWS_CASE(9)
    MOE_SUM_ROWS_CASE(10)
    MOE_SUM_ROWS_CASE(11)
    MOE_SUM_ROWS_CASE(12)
#undef MOE_SUM_ROWS_CASE
    static_assert(12 == kMaxRowsPerToken, "one instantiation per row count");
    default: return cudaErrorInvalidValue;
  }
  return e;
}

cudaError_t launch_dw_reduce(const float* partial, const int32_t* dest, int R, int nt, float* dw, int* err,
                             cudaStream_t s) {
  TraceScope trace_scope(MOE_K_DW_REDUCE, s);
  return launch_pdl(dw_reduce_kernel, dim3(ceil_div(R, 256)), dim3(256), 0, s, partial, dest, R, nt, dw, err);
}

cudaError_t launch_route_bwd(const float* logits, const int32_t* topk_idx, const float* topk_w, const float* dw,
                             int T, int E, int k, int renorm, float* dlogits, int* err, cudaStream_t s) {
  TraceScope trace_scope(MOE_K_ROUTE_BWD, s);
  const int blocks = min(ceil_div(T, 8), num_sms() * 8);
  cudaError_t e;
  if (E <= 32)
    e = launch_pdl(route_bwd_kernel<1>, dim3(blocks), dim3(256), 0, s, logits, topk_idx, topk_w, dw, T, E, k,
                   renorm, dlogits, err);
  else if (E <= 64)
    e = launch_pdl(route_bwd_kernel<2>, dim3(blocks), dim3(256), 0, s, logits, topk_idx, topk_w, dw, T, E, k,
                   renorm, dlogits, err);
  else if (E <= 128)
    e = launch_pdl(route_bwd_kernel<4>, dim3(blocks), dim3(256), 0, s, logits, topk_idx, topk_w, dw, T, E, k,
                   renorm, dlogits, err);
  else
    e = launch_pdl(route_bwd_kernel<8>, dim3(blocks), dim3(256), 0, s, logits, topk_idx, topk_w, dw, T, E, k,
                   renorm, dlogits, err);
  return e;
}

// Loads the modules of the kernels moe_dispatch runs (histogram, scan,
// scatter, row gather) if the runtime has not loaded them yet: under lazy
// module loading a kernel's module is loaded, and its device memory set up,
// on first use, and asking for a kernel's attributes is such a use.
cudaError_t preload_dispatch_kernels() {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, hist_kernel);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, scan_kernel);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, scatter_kernel);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, gather_rows_bf16_kernel);
  return e;
}

}  // namespace moe

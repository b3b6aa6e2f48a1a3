#pragma once
// Tile machinery shared by the persistent grouped GEMM and the forward MegaKernel:
// persistent grouped GEMM over ragged expert segments on tcgen05 tensor cores.
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
// Design (one CTA per SM, 192 threads):
//   warp 0      TMA producer: 128B-swizzled tiles of A (128 x 64) and B
//               (256 x 64) into a 4-stage shared-memory ring (48 KB/stage).
//   warp 1      allocates 512 TMEM columns, issues tcgen05.mma
//               (M=128, N=256, K=16, bf16 -> fp32) from one lane, commits
//               to mbarriers; a ragged-K tail is zeroed in shared memory.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (one TMEM lane per
//               thread = one output row), fused elementwise work, stores.
//   The accumulator is double-buffered in TMEM (2 x 256 columns) so the
//   epilogue of tile i overlaps the main loop of tile i+1.
// Tiles are taken in a static round-robin over CTAs; every output element is
// produced by exactly one tile with a fixed K order.
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

constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBBytes = kBN * kBK * 2;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 48 KB
constexpr int kBoxBytes = 64 * 64 * 2;          // one MN-major box: 64 x 64 bf16
constexpr int kMaxSeg = 256 + 4;
constexpr int kEpiWarps = 8;  // two epilogue warps per TMEM lane quadrant, one per half of the columns
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kTmemCols = 512;

struct GemmParams {
  CUtensorMap tmA0, tmA1, tmB0, tmB1;
  int T, d, f, E, k, S, R;
  int N;      // output columns per expert
  int Mw;     // ragged-K kinds: output rows per expert
  int K;      // ragged-M kinds: reduction length
  int nt_dh;  // dH: column tiles per row (number of partial dot products)
  const int32_t* offsets;
  const int32_t* row_slot;
  const float* topk_w;
  const uint16_t* aux_ab;
  const uint16_t* aux_h;
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
};

struct SharedState {
  uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], drain;
  uint32_t tmem_base;
  int abort;
  int nseg;
  int total_tiles;
  int seg_row0[kMaxSeg];
  int seg_rows[kMaxSeg];
  int prefix[kMaxSeg + 1];
};

constexpr int kSmemBytes = 1024 + kStages * kStageBytes + static_cast<int>(sizeof(SharedState));

struct TileInfo {
  int seg, m0, n0, rows, grow0, nkb;
  bool shared;
};

// Bounded wait that ignores the abort flag (used to drain in-flight copies).
__device__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

template <int KIND>
__device__ __forceinline__ int tiles_of(const GemmParams& p, int rows) {
  using Tr = Traits<KIND>;
  const int ntn = (p.N + Tr::BNE - 1) / Tr::BNE;
  if constexpr (Tr::RAGGED_K)
    return ((p.Mw + kBM - 1) / kBM) * ntn;
  else
    return ((rows + kBM - 1) / kBM) * ntn;
}

// Segment table: routed expert e owns GEMM rows [offsets[e], offsets[e+1]);
// shared expert s owns [R + s*T, R + (s+1)*T).  prefix[] counts tiles.
template <int KIND>
__device__ void build_segments(const GemmParams& p, SharedState& ss) {
  const int nseg = p.E + p.S;
  for (int s = threadIdx.x; s < nseg; s += blockDim.x) {
    int r0, n;
    if (s < p.E) {
      r0 = p.offsets[s];
      n = p.offsets[s + 1] - r0;
    } else {
      r0 = p.R + (s - p.E) * p.T;
      n = p.T;
    }
    ss.seg_row0[s] = r0;
    ss.seg_rows[s] = n;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (nseg + 31) / 32;
    const int lo = min(nseg, lane * per), hi = min(nseg, lo + per);
    int local = 0;
    for (int s = lo; s < hi; ++s) local += tiles_of<KIND>(p, ss.seg_rows[s]);
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    int run = incl - local;
    for (int s = lo; s < hi; ++s) {
      ss.prefix[s] = run;
      run += tiles_of<KIND>(p, ss.seg_rows[s]);
    }
    if (lane == 31) {
      ss.prefix[nseg] = incl;
      ss.total_tiles = incl;
      ss.nseg = nseg;
    }
  }
  __syncthreads();
}

template <int KIND>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, const SharedState& ss, int tile) {
  using Tr = Traits<KIND>;
  int lo = 0, hi = ss.nseg;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ss.prefix[mid] <= tile)
      lo = mid;
    else
      hi = mid;
  }
  TileInfo t;
  t.seg = lo;
  t.shared = lo >= p.E;
  const int local = tile - ss.prefix[lo];
  const int ntn = (p.N + Tr::BNE - 1) / Tr::BNE;
  const int mb = local / ntn, nb = local - mb * ntn;
  t.m0 = mb * kBM;
  t.n0 = nb * Tr::BNE;
  if constexpr (Tr::RAGGED_K) {
    t.rows = ss.seg_rows[lo];
    t.grow0 = ss.seg_row0[lo];
    t.nkb = (t.rows + kBK - 1) / kBK;
  } else {
    t.rows = min(kBM, ss.seg_rows[lo] - t.m0);
    t.grow0 = ss.seg_row0[lo] + t.m0;
    t.nkb = p.K / kBK;
  }
  return t;
}

// One stage of TMA loads (48 KB in every kind).
template <int KIND>
__device__ __forceinline__ void issue_loads(const GemmParams& p, const TileInfo& t, int kb, uint8_t* sA,
                                            uint8_t* sB, uint64_t* bar) {
  const int kk = kb * kBK;
  if constexpr (KIND == kG1) {
    tma_load_2d(sA, t.shared ? &p.tmA1 : &p.tmA0, bar, kk, t.shared ? t.m0 : t.grow0);
    tma_load_2d(sB, &p.tmB0, bar, kk, t.seg * p.f + t.n0);
    tma_load_2d(sB + kBBytes / 2, &p.tmB1, bar, kk, t.seg * p.f + t.n0);
  } else if constexpr (KIND == kG2) {
    tma_load_2d(sA, &p.tmA0, bar, kk, t.grow0);
    tma_load_2d(sB, &p.tmB0, bar, kk, t.seg * p.d + t.n0);
  } else if constexpr (KIND == kDH) {
    tma_load_2d(sA, t.shared ? &p.tmA1 : &p.tmA0, bar, kk, t.shared ? t.m0 : t.grow0);
#pragma unroll
    for (int i = 0; i < 4; ++i) tma_load_2d(sB + i * kBoxBytes, &p.tmB0, bar, t.n0 + 64 * i, t.seg * p.d + kk);
  } else if constexpr (KIND == kDX) {
    tma_load_2d(sA, &p.tmA0, bar, kk, t.grow0);
    const bool second = kk >= p.f;
    const int krow = t.seg * p.f + (second ? kk - p.f : kk);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      tma_load_2d(sB + i * kBoxBytes, second ? &p.tmB1 : &p.tmB0, bar, t.n0 + 64 * i, krow);
  } else if constexpr (KIND == kDW13) {
#pragma unroll
    for (int i = 0; i < 2; ++i) tma_load_2d(sA + i * kBoxBytes, &p.tmA0, bar, t.m0 + 64 * i, t.grow0 + kk);
    const int brow = t.shared ? kk : t.grow0 + kk;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      tma_load_2d(sB + i * kBoxBytes, t.shared ? &p.tmB1 : &p.tmB0, bar, t.n0 + 64 * i, brow);
  } else {  // kDW2
    const int arow = t.shared ? kk : t.grow0 + kk;
#pragma unroll
    for (int i = 0; i < 2; ++i)
      tma_load_2d(sA + i * kBoxBytes, t.shared ? &p.tmA1 : &p.tmA0, bar, t.m0 + 64 * i, arow);
#pragma unroll
    for (int i = 0; i < 4; ++i) tma_load_2d(sB + i * kBoxBytes, &p.tmB0, bar, t.n0 + 64 * i, t.grow0 + kk);
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void store_f32x32(float* dst, const uint32_t (&v)[32], float scale) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    d4[i] = make_float4(scale * __uint_as_float(v[4 * i]), scale * __uint_as_float(v[4 * i + 1]),
                        scale * __uint_as_float(v[4 * i + 2]), scale * __uint_as_float(v[4 * i + 3]));
}
__device__ __forceinline__ void store_zero_f32x32(float* dst) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) d4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Epilogue of one tile for the thread owning tile row `row` (TMEM lane).
template <int KIND>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const TileInfo& t, int row, int half,
                                              uint32_t tacc) {
  if constexpr (KIND == kG1) {
    // Columns [0,128) hold a (gate), [128,256) hold b (up) for outputs n0..n0+127.
    const bool ok = row < t.rows;
    const size_t grow = static_cast<size_t>(t.grow0) + row;
    uint16_t* H = static_cast<uint16_t*>(p.out0);
    uint16_t* AB = static_cast<uint16_t*>(p.out1);
#pragma unroll 1
    for (int c = 2 * half; c < 2 * half + 2; ++c) {
      const int n = t.n0 + 32 * c;
      if (n >= p.f) break;
      uint32_t a[32], b[32];
      tmem_ld_32x32(tacc + 32 * c, a);
      tmem_ld_32x32(tacc + 128 + 32 * c, b);
      tmem_ld_wait();
      if (ok) {
        uint32_t hp[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a0 = __uint_as_float(a[2 * i]), a1 = __uint_as_float(a[2 * i + 1]);
          const float b0 = __uint_as_float(b[2 * i]), b1 = __uint_as_float(b[2 * i + 1]);
          const float h0 = a0 / (1.f + expf(-a0)) * b0;
          const float h1 = a1 / (1.f + expf(-a1)) * b1;
          hp[i] = pack_bf16(h0, h1);
        }
        uint4* dst = reinterpret_cast<uint4*>(H + grow * p.f + n);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hp[4 * i], hp[4 * i + 1], hp[4 * i + 2], hp[4 * i + 3]);
        if (AB) {
          uint4* da = reinterpret_cast<uint4*>(AB + grow * 2 * p.f + n);
          uint4* db = reinterpret_cast<uint4*>(AB + grow * 2 * p.f + p.f + n);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            da[i] = make_uint4(pack_bf16(__uint_as_float(a[8 * i]), __uint_as_float(a[8 * i + 1])),
                               pack_bf16(__uint_as_float(a[8 * i + 2]), __uint_as_float(a[8 * i + 3])),
                               pack_bf16(__uint_as_float(a[8 * i + 4]), __uint_as_float(a[8 * i + 5])),
                               pack_bf16(__uint_as_float(a[8 * i + 6]), __uint_as_float(a[8 * i + 7])));
            db[i] = make_uint4(pack_bf16(__uint_as_float(b[8 * i]), __uint_as_float(b[8 * i + 1])),
                               pack_bf16(__uint_as_float(b[8 * i + 2]), __uint_as_float(b[8 * i + 3])),
                               pack_bf16(__uint_as_float(b[8 * i + 4]), __uint_as_float(b[8 * i + 5])),
                               pack_bf16(__uint_as_float(b[8 * i + 6]), __uint_as_float(b[8 * i + 7])));
          }
        }
      }
    }
  } else if constexpr (KIND == kG2 || KIND == kDX) {
    const bool ok = row < t.rows;
    const size_t grow = static_cast<size_t>(t.grow0) + row;
    float w = 1.f;
    if constexpr (KIND == kG2)
      if (ok && !t.shared) w = p.topk_w[p.row_slot[grow]];
    float* out = static_cast<float*>(p.out0);
#pragma unroll 1
    for (int c = 4 * half; c < 4 * half + 4; ++c) {
      const int n = t.n0 + 32 * c;
      if (n >= p.d) break;
      uint32_t v[32];
      tmem_ld_32x32(tacc + 32 * c, v);
      tmem_ld_wait();
      if (ok) store_f32x32(out + grow * p.d + n, v, w);
    }
  } else if constexpr (KIND == kDH) {
    const bool ok = row < t.rows;
    const size_t grow = static_cast<size_t>(t.grow0) + row;
    float w = 1.f;
    if (ok && !t.shared) w = p.topk_w[p.row_slot[grow]];
    uint16_t* dAB = static_cast<uint16_t*>(p.out0);
    uint16_t* Hw = static_cast<uint16_t*>(p.out1);
    float dot = 0.f;
#pragma unroll 1
    for (int c = 4 * half; c < 4 * half + 4; ++c) {
      const int n = t.n0 + 32 * c;
      if (n >= p.f) break;
      uint32_t g[32];
      tmem_ld_32x32(tacc + 32 * c, g);
      tmem_ld_wait();
      if (ok) {
        const uint4* pa = reinterpret_cast<const uint4*>(p.aux_ab + grow * 2 * p.f + n);
        const uint4* pb = reinterpret_cast<const uint4*>(p.aux_ab + grow * 2 * p.f + p.f + n);
        const uint4* ph = reinterpret_cast<const uint4*>(p.aux_h + grow * p.f + n);
        uint4* oa = reinterpret_cast<uint4*>(dAB + grow * 2 * p.f + n);
        uint4* ob = reinterpret_cast<uint4*>(dAB + grow * 2 * p.f + p.f + n);
        uint4* oh = reinterpret_cast<uint4*>(Hw + grow * p.f + n);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 av = __ldg(pa + q), bv = __ldg(pb + q), hv = __ldg(ph + q);
          const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
          const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
          const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
          uint32_t ra[4], rb[4], rh[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float dA2[2], dB2[2], hw2[2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const float a = half ? bf16_hi(aw[u]) : bf16_lo(aw[u]);
              const float b = half ? bf16_hi(bw[u]) : bf16_lo(bw[u]);
              const float h = half ? bf16_hi(hw[u]) : bf16_lo(hw[u]);
              const float graw = __uint_as_float(g[8 * q + 2 * u + half]);
              dot += graw * h;
              const float dH = w * graw;
              const float s = 1.f / (1.f + expf(-a));
              dA2[half] = dH * b * s * (1.f + a * (1.f - s));
              dB2[half] = dH * (a * s);
              hw2[half] = w * h;
            }
            ra[u] = pack_bf16(dA2[0], dA2[1]);
            rb[u] = pack_bf16(dB2[0], dB2[1]);
            rh[u] = pack_bf16(hw2[0], hw2[1]);
          }
          oa[q] = make_uint4(ra[0], ra[1], ra[2], ra[3]);
          ob[q] = make_uint4(rb[0], rb[1], rb[2], rb[3]);
          oh[q] = make_uint4(rh[0], rh[1], rh[2], rh[3]);
        }
      }
    }
    if (ok && !t.shared) p.out_partial[(grow * p.nt_dh + t.n0 / kBN) * 2 + half] = dot;
  } else if constexpr (KIND == kDW13) {
    // Output row m of the stacked [dW1_e ; dW3_e] (2f rows), columns n (d).
    const int m = t.m0 + row;
    float* out = (m < p.f) ? static_cast<float*>(p.out0) + (static_cast<size_t>(t.seg) * p.f + m) * p.d
                           : static_cast<float*>(p.out1) + (static_cast<size_t>(t.seg) * p.f + (m - p.f)) * p.d;
#pragma unroll 1
    for (int c = 4 * half; c < 4 * half + 4; ++c) {
      const int n = t.n0 + 32 * c;
      if (n >= p.d) break;
      if (t.nkb == 0) {
        store_zero_f32x32(out + n);
        continue;
      }
      uint32_t v[32];
      tmem_ld_32x32(tacc + 32 * c, v);
      tmem_ld_wait();
      store_f32x32(out + n, v, 1.f);
    }
  } else {  // kDW2: output row m (d) of dW2_e, columns n (f)
    const int m = t.m0 + row;
    const bool ok = m < p.d;
    float* out = static_cast<float*>(p.out0) + (static_cast<size_t>(t.seg) * p.d + m) * p.f;
#pragma unroll 1
    for (int c = 4 * half; c < 4 * half + 4; ++c) {
      const int n = t.n0 + 32 * c;
      if (n >= p.f) break;
      if (t.nkb == 0) {
        if (ok) store_zero_f32x32(out + n);
        continue;
      }
      uint32_t v[32];
      tmem_ld_32x32(tacc + 32 * c, v);
      tmem_ld_wait();
      if (ok) store_f32x32(out + n, v, 1.f);
    }
  }
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

// Row-major bf16 matrix [outer, inner] seen as 2D tiles of box_outer rows x
// box_inner (= 64, one 128-byte swizzle span) columns; out-of-range reads
// fill zeros.
bool map2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
           uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !base || inner == 0 || outer == 0) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// ---------------------------------------------------------- per-tile roles
// Shared by the grouped GEMM kernel and the MegaKernel, so a tile's MMA
// sequence and epilogue arithmetic are the same code in both.

__device__ __forceinline__ void init_gemm_barriers(SharedState& ss) {
  for (int s = 0; s < kStages; ++s) {
    mbar_init(&ss.full[s], 1);
    mbar_init(&ss.empty[s], 1);
  }
  for (int a = 0; a < 2; ++a) {
    mbar_init(&ss.tfull[a], 1);
    mbar_init(&ss.tempty[a], kEpiWarps);
  }
  mbar_init(&ss.drain, 1);
  ss.abort = 0;
}

// Producer lane: every K block of one tile through the stage ring.
struct ProducerState {
  int stage = 0;
  uint32_t phase = 0, filled = 0, fill_par = 0;
};

template <int KIND>
__device__ __forceinline__ bool produce_tile(const GemmParams& p, const TileInfo& t, SharedState& ss, uint8_t* smem,
                                             ProducerState& ps, volatile int* abort, int where) {
  for (int kb = 0; kb < t.nkb; ++kb) {
    if (!mbar_wait(&ss.empty[ps.stage], ps.phase ^ 1, abort, p.err, where)) return false;
    uint8_t* sA = smem + ps.stage * kStageBytes;
    mbar_arrive_expect_tx(&ss.full[ps.stage], kStageBytes);
    issue_loads<KIND>(p, t, kb, sA, sA + kABytes, &ss.full[ps.stage]);
    ps.filled |= 1u << ps.stage;
    ps.fill_par = (ps.fill_par & ~(1u << ps.stage)) | (ps.phase << ps.stage);
    if (++ps.stage == kStages) {
      ps.stage = 0;
      ps.phase ^= 1;
    }
  }
  return true;
}

// Lets every copy the producer issued land before the CTA may exit.
__device__ __forceinline__ void producer_drain(SharedState& ss, const ProducerState& ps) {
  for (int s = 0; s < kStages; ++s)
    if (ps.filled & (1u << s)) mbar_wait_drain(&ss.full[s], (ps.fill_par >> s) & 1);
}

// MMA warp: one tile into TMEM accumulator buffer `acc`; lane 0 issues.
struct MmaState {
  int stage = 0, it = 0;
  uint32_t phase = 0;
  bool issued = false;
};

template <int KIND>
__device__ __forceinline__ bool mma_tile(const GemmParams& p, const TileInfo& t, SharedState& ss, uint8_t* smem,
                                         uint32_t tmem, MmaState& ms, volatile int* abort, int where) {
  using Tr = Traits<KIND>;
  constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, Tr::A_MN ? 1 : 0, Tr::B_MN ? 1 : 0);
  const int lane = threadIdx.x & 31;
  const int acc = ms.it & 1;
  const uint32_t aph = (ms.it >> 1) & 1;
  ++ms.it;
  if (!mbar_wait(&ss.tempty[acc], aph ^ 1, abort, p.err, where)) return false;
  tc_fence_after();
  const uint32_t dtm = tmem + acc * kBN;
  for (int kb = 0; kb < t.nkb; ++kb) {
    if (!mbar_wait(&ss.full[ms.stage], ms.phase, abort, p.err, where | (1 << 20))) return false;
    tc_fence_after();
    uint8_t* sA = smem + ms.stage * kStageBytes;
    uint8_t* sB = sA + kABytes;
    if constexpr (Tr::RAGGED_K) {
      const int kvalid = t.rows - kb * kBK;
      if (kvalid < kBK) {  // rows past the segment end must not contribute
        const int per_box = (kBK - kvalid) * 8;
        for (int idx = lane; idx < 6 * per_box; idx += 32) {
          const int box = idx / per_box, rem = idx - box * per_box;
          uint8_t* bb = (box < 2) ? sA + box * kBoxBytes : sB + (box - 2) * kBoxBytes;
          reinterpret_cast<uint4*>(bb + (kvalid + rem / 8) * 128)[rem & 7] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
    }
    if (lane == 0) {
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
      for (int k4 = 0; k4 < kBK / 16; ++k4) {
        const uint64_t ad = Tr::A_MN ? smem_desc_sw128(a0 + k4 * 2048, kBoxBytes, 1024)
                                     : smem_desc_sw128(a0 + k4 * 32, 16, 1024);
        const uint64_t bd = Tr::B_MN ? smem_desc_sw128(b0 + k4 * 2048, kBoxBytes, 1024)
                                     : smem_desc_sw128(b0 + k4 * 32, 16, 1024);
        umma_bf16(dtm, ad, bd, kIdesc, (kb | k4) != 0 ? 1u : 0u);
      }
      umma_commit(&ss.empty[ms.stage]);
      ms.issued = true;
    }
    __syncwarp();
    if (++ms.stage == kStages) {
      ms.stage = 0;
      ms.phase ^= 1;
    }
  }
  if (lane == 0) umma_commit(&ss.tfull[acc]);
  __syncwarp();
  return true;
}

// Waits for the tensor core before TMEM is released on an aborted run.
__device__ __forceinline__ void mma_drain(SharedState& ss, const MmaState& ms) {
  if ((threadIdx.x & 31) == 0 && ms.issued) {
    umma_commit(&ss.drain);
    mbar_wait_drain(&ss.drain, 0);
  }
  __syncwarp();
}

// Epilogue warps (2..5): one tile out of TMEM buffer `it & 1`.
template <int KIND>
__device__ __forceinline__ bool epilogue_step(const GemmParams& p, const TileInfo& t, SharedState& ss, uint32_t tmem,
                                              int& it, volatile int* abort, int where) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lanes [32q, 32q+32) are reachable from this warp
  const int acc = it & 1;
  const uint32_t aph = (it >> 1) & 1;
  ++it;
  if (!mbar_wait(&ss.tfull[acc], aph, abort, p.err, where)) return false;
  tc_fence_after();
  const int half = (warp - 2) >> 2;  // columns [128*half, 128*half + 128) of the accumulator
  epilogue_tile<KIND>(p, t, q * 32 + lane, half, tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN);
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&ss.tempty[acc]);
  return true;
}

// Tensor maps and pointers of one GEMM kind.
template <int KIND>
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
    p.N = a.f;
    p.K = a.d;
    p.out0 = a.H_out;
    p.out1 = a.AB_out;
  } else if constexpr (KIND == kG2) {
    ok &= map2d(&p.tmA0, a.H, f, Rs, 64, 128);
    ok &= map2d(&p.tmB0, a.W2, f, nexp * d, 64, 256);
    p.N = a.d;
    p.K = a.f;
    p.out0 = a.Op_out;
  } else if constexpr (KIND == kDH) {
    ok &= map2d(&p.tmA0, a.G, d, R, 64, 128);
    ok &= map2d(&p.tmA1, a.dy, d, T, 64, 128);
    ok &= map2d(&p.tmB0, a.W2, f, nexp * d, 64, 64);
    p.N = a.f;
    p.K = a.d;
    p.aux_ab = a.AB;
    p.aux_h = a.H;
    p.out0 = a.dAB_out;
    p.out1 = a.Hw_out;
    p.out_partial = a.partial_out;
  } else if constexpr (KIND == kDX) {
    ok &= map2d(&p.tmA0, a.dAB, 2 * f, Rs, 64, 128);
    ok &= map2d(&p.tmB0, a.W1, d, nexp * f, 64, 64);
    ok &= map2d(&p.tmB1, a.W3, d, nexp * f, 64, 64);
    p.N = a.d;
    p.K = 2 * a.f;
    p.out0 = a.dXp_out;
  } else if constexpr (KIND == kDW13) {
    ok &= map2d(&p.tmA0, a.dAB, 2 * f, Rs, 64, 64);
    ok &= map2d(&p.tmB0, a.Xp, d, R, 64, 64);
    ok &= map2d(&p.tmB1, alt(a.x, a.Xp), d, a.x ? T : R, 64, 64);
    p.Mw = 2 * a.f;
    p.N = a.d;
    p.out0 = a.dW1_out;
    p.out1 = a.dW3_out;
  } else {
    ok &= map2d(&p.tmA0, a.G, d, R, 64, 64);
    ok &= map2d(&p.tmA1, a.dy, d, T, 64, 64);
    ok &= map2d(&p.tmB0, a.Hw, f, Rs, 64, 64);
    p.Mw = a.d;
    p.N = a.f;
    p.out0 = a.dW2_out;
  }
  return ok;
}
}  // namespace
}  // namespace moe

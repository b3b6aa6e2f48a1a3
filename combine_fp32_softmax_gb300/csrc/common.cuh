// Shared definitions of the CUDA library: error recording, workspace layout,
// tile constants.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/moe.h"

namespace moe {

// Error codes as stored in the device error word (same values as moe.h).
constexpr int MOE_ERR_NONFINITE_CODE = MOE_ERR_NONFINITE;
constexpr int MOE_ERR_TIMEOUT_CODE = MOE_ERR_TIMEOUT;

// Longest any spin in this library waits before giving up (1 s).  Normal
// waits last microseconds; the limit only turns a bug into an error code
// instead of a hung GPU.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

#ifdef __CUDACC__
// First error wins: code in err[0], detail in err[1].
__device__ __forceinline__ void record_error(int* err, int code, int info) {
  if (atomicCAS(err, 0, code) == 0) atomicExch(err + 1, info);
}
#endif

// Checks of the debug build (compiled with -DMOE_DEBUG; the release build
// compiles them out).  A failed check records MOE_ERR_ARG with the site and
// a detail in the device error word, info = site << 24 | (detail & 0xFFFFFF);
// the kernel then skips the access it guards.  No check traps: the launch
// still returns normally and the context stays usable.
#ifdef MOE_DEBUG
constexpr bool kDebug = true;
#else
constexpr bool kDebug = false;
#endif
enum DebugSite : int {
  kDbgGatherRow = 0x41,     // gathered row index outside the source rows
  kDbgScatterRow = 0x42,    // destination row outside the gathered rows
  kDbgSumRow = 0x43,        // summed row outside the rows
  kDbgDwReduce = 0x44,      // dw partial row outside the routed rows
  kDbgRouteBwd = 0x45,      // expert index outside [0, E)
  kDbgPermRow = 0x46,       // permutation row outside [0, R)
  kDbgSegments = 0x50,      // + GEMM kind: segment table not monotone / not ending at R
  kDbgTmaCoord = 0x58,      // + GEMM kind: TMA box start misaligned or negative
  kDbgEpiRow = 0x60,        // + GEMM kind: epilogue row outside the GEMM rows, or its slot outside [0, R)
  kDbgMegaGather = 0x68,    // MegaKernel gather: token outside [0, T)
  kDbgMegaCombine = 0x69,   // MegaKernel token sum: row outside the rows
};
#ifdef __CUDACC__
__device__ __forceinline__ bool debug_ok(bool cond, int* err, int site, long long detail) {
  if constexpr (kDebug) {
    if (!cond && err) record_error(err, MOE_ERR_ARG, site << 24 | static_cast<int>(detail & 0xFFFFFF));
    return cond;
  } else {
    return true;
  }
}
#endif

// Words of the 64-byte error region (int index) that hold the grid barrier
// of the fused routing + permutation kernel: the arrival count (back to 0
// after every completed barrier) and the generation.  moe_ws_init zeroes
// them with the error word.
constexpr int kErrBarrierWord = 8;
// Words of the error region (which spans 256 bytes) that hold each grouped
// GEMM kind's tile-ticket counter and finished-CTA count, two per kind from
// this word on; both are back at 0 after every complete launch.
constexpr int kErrSchedWord = 16;
constexpr int kErrRegionBytes = 256;

// Router / permutation: tokens per histogram block (the router and the fused
// routing kernel run one warp per token, the stand-alone scatter 8 warps of 4
// tokens).  Small blocks give the latency-bound router enough warps; the
// per-block histogram the scan walks has E * ceil(T / 32) entries.
constexpr int kRouteTokensPerBlock = 32;

// Grouped GEMM tile: 128 rows x 256 accumulator columns, K staged 64 at a
// time (one 128-byte swizzle atom of bf16).
constexpr int kBM = 128;
// Smallest rows per MegaKernel gather task (the counter region is sized for
// it): small tasks spread the gather (a bulk load per row from one lane)
// over many CTAs when there are few rows.
constexpr int kMegaGatherRows = 32;
constexpr int kBN = 256;
constexpr int kBK = 64;

inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Launch attribute of programmatic dependent launch: the kernel may be
// scheduled while the previous kernel on the stream still runs (it calls
// griddep_wait() before touching global data).
inline void set_pdl_attr(cudaLaunchAttribute& a) {
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  set_pdl_attr(attr[0]);
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Offsets of the regions inside the caller's workspace (bytes from ws).
struct WsLayout {
  size_t err, hist, base, counts, offsets, dest, row_token, row_slot;
  size_t Xp, AB, Hw, Op, G, dAB, dXp, partial, dw, mk;
  size_t total;
  int nb_route;  // router/permutation blocks
  int nt_dh;     // column tiles of the dH GEMM (partial dot products per row)
  int mk_ints;   // ints in the MegaKernel counter region
};

inline WsLayout ws_layout(const moe_cfg& c) {
  WsLayout L{};
  const size_t T = c.T, d = c.d_model, f = c.d_ff, E = c.E, k = c.k, S = c.n_shared;
  const size_t R = T * k, Rs = R + S * T;
  L.nb_route = ceil_div(c.T, kRouteTokensPerBlock);
  L.nt_dh = ceil_div(c.d_ff, kBN);  // dw partial dots: one per 256-column tile of a row
  // MegaKernel counters: cursor + 3 phase counters, one readiness counter
  // per gathered row block (kMegaGatherRows rows), one per first-GEMM m-tile
  // (bounded by the m-tiles of every segment), padding.
  const size_t mtiles_max = R / kBM + E + S * static_cast<size_t>(ceil_div(c.T, kBM)) + 2;
  L.mk_ints = static_cast<int>(16 + ceil_div(static_cast<long long>(R), kMegaGatherRows) + mtiles_max + 16);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.err = take(kErrRegionBytes);
  L.hist = take(sizeof(int) * E * L.nb_route);
  L.base = take(sizeof(int) * E * L.nb_route);
  L.counts = take(sizeof(int) * E);
  L.offsets = take(sizeof(int) * (E + 1));
  L.dest = take(sizeof(int) * R);
  L.row_token = take(sizeof(int) * R);
  L.row_slot = take(sizeof(int) * R);
  L.Xp = take(2 * R * d);
  L.AB = take(2 * Rs * 2 * f);
  L.Hw = take(2 * Rs * f);
  L.Op = take(4 * Rs * d);
  L.G = take(2 * R * d);
  L.dAB = take(2 * Rs * 2 * f);
  L.dXp = take(4 * Rs * d);
  L.partial = take(4 * R * L.nt_dh);  // one partial dot per (row, 256-column tile)
  L.dw = take(4 * T * k);
  L.mk = take(sizeof(int) * L.mk_ints);
  L.total = o;
  return L;
}

}  // namespace moe

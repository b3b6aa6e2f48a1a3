// Persistent grouped GEMM over ragged expert segments on tcgen05 tensor cores
// (one kernel per GEMM kind; the tile machinery is in gemm_tiles.cuh).
//
// Warp roles, shared-memory ring, TMEM double buffering and the staged TMA
// epilogues are described in gemm_tiles.cuh.  Tiles are taken in a static
// round-robin over CTAs; every output element is produced by exactly one
// tile with a fixed K order.
#include "gemm_tiles.cuh"

namespace moe {
namespace {

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
  using Tr = Traits<KIND>;
  constexpr int NST = Tr::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stg_base = smem + NST * kStageBytes;  // epilogue staging, Tr::EPI_BYTES per epilogue warp
  SharedState& ss = *reinterpret_cast<SharedState*>(stg_base + kEpiWarps * Tr::EPI_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    init_gemm_barriers(ss);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ss.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  build_segments<KIND>(p, ss);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ss.tmem_base;
  const int total = ss.total_tiles;
  volatile int* abort = &ss.abort;
  const int where0 = (KIND + 1) << 24;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.tmA0);
      tma_prefetch_desc(&p.tmB0);
      ProducerState ps;
      for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x)
        if (!produce_tile<KIND, NST>(p, decode_tile<KIND>(p, ss, tile), ss, smem, ps, abort, where0 | tile)) break;
      if (*abort) producer_drain(ss, ps);
    }
  } else if (warp == 1) {
    MmaState ms;
    for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x)
      if (!mma_tile<KIND, NST>(p, decode_tile<KIND>(p, ss, tile), ss, smem, tmem, ms, abort,
                               where0 | (2 << 20) | tile))
        break;
    if (*abort) mma_drain(ss, ms);
  } else {
    EpiState es;
    uint8_t* stg = stg_base + (warp & 3) * Tr::EPI_BYTES;
    for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x)
      if (!epilogue_step<KIND>(p, decode_tile<KIND>(p, ss, tile), ss, tmem, stg, es, abort,
                               where0 | (4 << 20) | tile))
        break;
    epilogue_drain(ss, es);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int KIND>
int launch_kind(const GemmArgs& a, cudaStream_t s, int grid_override) {
  GemmParams p;
  if (!fill_params<KIND>(a, p)) return MOE_ERR_CUDA;
  constexpr int kSmem = smem_bytes<KIND>();
  static_assert(kSmem <= 232448, "shared memory budget of one CTA");
  if (cudaFuncSetAttribute(grouped_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const int grid = grid_override > 0 ? grid_override : num_sms();
  constexpr int kTrace[6] = {MOE_K_GEMM1, MOE_K_GEMM2, MOE_K_GEMM_DH, MOE_K_GEMM_DX, MOE_K_GEMM_DW13, MOE_K_GEMM_DW2};
  TraceScope trace_scope(kTrace[KIND], s);
  grouped_gemm_kernel<KIND><<<grid, kThreads, kSmem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

int launch_gemm(GemmKind kind, const GemmArgs& a, cudaStream_t s, int grid_override) {
  switch (kind) {
    case kG1: return launch_kind<kG1>(a, s, grid_override);
    case kG2: return launch_kind<kG2>(a, s, grid_override);
    case kDH: return launch_kind<kDH>(a, s, grid_override);
    case kDX: return launch_kind<kDX>(a, s, grid_override);
    case kDW13: return launch_kind<kDW13>(a, s, grid_override);
    case kDW2: return launch_kind<kDW2>(a, s, grid_override);
  }
  return MOE_ERR_ARG;
}

}  // namespace moe

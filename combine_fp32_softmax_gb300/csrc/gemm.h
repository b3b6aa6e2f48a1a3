// Grouped GEMM family over ragged expert segments (host launchers).
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"

namespace moe {

enum GemmKind : int {
  kG1 = 0,    // forward gate/up: A = Xp (x for shared rows), B = [W1 | W3] -> Hw = w * h (+ [a|b])
  kG2 = 1,    // forward down:    A = Hw, B = W2 -> O' = w * o (fp32)
  kDH = 2,    // backward dH:     A = G (dy for shared rows), B = W2 (MN-major) -> dAB, dw partials
  kDX = 3,    // backward dX:     A = dAB, B = [W1 ; W3] (MN-major) -> dXp (fp32)
  kDW13 = 4,  // backward dW1/3:  A = dAB^T, B = Xp^T (x^T for shared), ragged K -> dW1, dW3 (fp32)
  kDW2 = 5,   // backward dW2:    A = G^T (dy^T for shared), B = Hw^T, ragged K -> dW2 (fp32)
};

// Pointers of one layer-level GEMM call.  Which are used depends on the kind.
struct GemmArgs {
  int T, d, f, E, k, S;
  const int32_t* offsets;
  const int32_t* row_slot;
  const float* topk_w;
  // operands (bf16)
  const uint16_t* Xp;
  const uint16_t* x;
  const uint16_t* W1;
  const uint16_t* W3;
  const uint16_t* W2;
  const uint16_t* AB;
  const uint16_t* G;
  const uint16_t* dy;
  const uint16_t* dAB;
  const uint16_t* Hw;
  // outputs
  uint16_t* Hw_out;
  uint16_t* AB_out;
  float* Op_out;
  uint16_t* dAB_out;
  float* partial_out;
  float* dXp_out;
  float* dW1_out;
  float* dW3_out;
  float* dW2_out;
  int* err;
};

// Returns MOE_OK or a negative MOE_ERR_* (tensor-map encoding or launch).
int launch_gemm(GemmKind kind, const GemmArgs& a, cudaStream_t s, int grid_override = 0);

// dX, dW1/dW3 and dW2 as one persistent launch with their tiles interleaved
// (same outputs, bit for bit, as the three separate launches).  CTA pairs
// when all three kinds run on pairs.
int launch_bwd_gemms(const GemmArgs& a, cudaStream_t s, int grid_override = 0);

// Bit k set: kind k runs on CTA pairs (256-row tiles); clear: one CTA per
// 128-row tile.  Returns the previous mask.
int set_gemm_pair_kinds(int mask);
// The current mask (as set_gemm_pair_kinds).
int gemm_pair_kinds();

// K blocks of each CTA's next tile that kind `kind` prefetches into L2 while
// loading the current one (0 = none, at most 64).  Returns the previous
// value, or -1 for an unknown kind.
int set_gemm_prefetch(GemmKind kind, int kblocks);

// Tile order of a ragged-K kind (kDW13, kDW2): 0 = longest segments first,
// 1 = the long segments' tiles interleaved with the short ones.  Returns
// the previous order, or -1 for another kind.
int set_gemm_tile_order(GemmKind kind, int order);

// Epilogue stores of an fp32-output kind (kG2, kDX, kDW13, kDW2): 0 = staged
// through shared memory and written by TMA, 1 = straight from registers.
// Returns the previous mode, or -1 for another kind.
int set_gemm_epilogue(GemmKind kind, int direct);

// Pipeline stages kind `kind` uses (0 or out of range: as many as fit; at
// least 2).  Returns the previous request, or -1 for an unknown kind.
int set_gemm_stages(GemmKind kind, int stages);
// Stages that fit for `kind` with `cta_group` CTAs per tile, with its
// current epilogue stores; the second form names the epilogue mode
// (1 = direct: no staging memory, so an fp32-output kind fits more).
int gemm_max_stages(GemmKind kind, int cta_group);
int gemm_max_stages(GemmKind kind, int cta_group, int direct);

// CTA pairs of `kind` that fit on the device at once (0 on error).
int gemm_pair_capacity(GemmKind kind);

}  // namespace moe

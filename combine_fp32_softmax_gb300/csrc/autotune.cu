// Measured autotuner for the grouped GEMMs: per GEMM kind, the tile shape
// (one CTA per 128 x 256 tile, or a CTA pair per 256 x 256 tile) and the
// depth of the next-tile L2 prefetch are chosen by timing the caller's own
// layer.  None of these choices changes any arithmetic, so results are the
// same bits before and after tuning.
//
// UniEP page ("Unified Expert-Parallel MoE MegaKernel for LLM Training"),
// section 3 (autotuning and the analytical model) names the step but gives no
// content; this is the plainest reading: measure the candidates on the
// workload and keep the fastest per kernel.
#include <cuda_runtime.h>

#include "common.cuh"
#include "gemm.h"

namespace {

constexpr int kKinds = 6;
constexpr int kTraceOf[kKinds] = {MOE_K_GEMM1,  MOE_K_GEMM2,     MOE_K_GEMM_DH,
                                  MOE_K_GEMM_DX, MOE_K_GEMM_DW13, MOE_K_GEMM_DW2};
constexpr int kDepths[] = {0, 4, 8};
constexpr int kNumDepths = sizeof(kDepths) / sizeof(kDepths[0]);
// A candidate replaces the one kept so far only if it is faster by more than
// this fraction (about the run-to-run spread of a kernel's time), so near
// ties keep the first candidate timed: CTA pairs without prefetch, the
// default.
constexpr double kMargin = 0.01;

}  // namespace

extern "C" int moe_autotune(const moe_cfg* cfg, const float* logits, const uint16_t* x, const uint16_t* W1,
                            const uint16_t* W3, const uint16_t* W2, const uint16_t* dy, float* y,
                            int32_t* topk_idx, float* topk_w, float* dx, float* dlogits, float* dW1, float* dW3,
                            float* dW2, void* ws, int reps, void* stream, moe_tune_result* out) {
  using namespace moe;
  if (!out || reps < 0) return MOE_ERR_ARG;
  if (reps == 0) reps = 2;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Previous settings, restored on any failure.
  const int prev_mask = set_gemm_pair_kinds(0);
  set_gemm_pair_kinds(prev_mask);
  int prev_depth[kKinds];
  for (int k = 0; k < kKinds; ++k) {
    prev_depth[k] = set_gemm_prefetch(static_cast<GemmKind>(k), 0);
    set_gemm_prefetch(static_cast<GemmKind>(k), prev_depth[k]);
  }
  // The backward's B/W overlap is off while timing: a weight-gradient GEMM
  // on the second stream would otherwise be charged its wait for the SMs
  // that dX holds.
  const int prev_overlap = moe_set_bwd_overlap(0);
  auto restore = [&]() {
    set_gemm_pair_kinds(prev_mask);
    for (int k = 0; k < kKinds; ++k) set_gemm_prefetch(static_cast<GemmKind>(k), prev_depth[k]);
    moe_trace_enable(0);
    moe_set_bwd_overlap(prev_overlap);
  };
  auto step = [&]() -> int {
    int rc = moe_layer_fwd(cfg, logits, x, W1, W3, W2, y, topk_idx, topk_w, ws, 0, stream);
    if (rc == MOE_OK)
      rc = moe_layer_bwd(cfg, dy, logits, x, W1, W3, W2, topk_idx, topk_w, ws, dx, dlogits, dW1, dW3, dW2, 3,
                         stream);
    return rc;
  };

  double best[kKinds];
  for (int k = 0; k < kKinds; ++k) best[k] = -1.0;
  for (int pi = 0; pi < 2; ++pi) {
    const int pair = 1 - pi;  // CTA pairs first
    for (int di = 0; di < kNumDepths; ++di) {
      set_gemm_pair_kinds(pair ? (1 << kKinds) - 1 : 0);
      for (int k = 0; k < kKinds; ++k) set_gemm_prefetch(static_cast<GemmKind>(k), kDepths[di]);
      moe_trace_enable(0);
      int rc = step();  // warm-up of this candidate (first launches set up tensor maps and attributes)
      if (rc == MOE_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = MOE_ERR_CUDA;
      if (rc == MOE_OK) {
        moe_trace_reset();
        moe_trace_enable(1);
        for (int r = 0; r < reps && rc == MOE_OK; ++r) rc = step();
        moe_trace_enable(0);
        if (rc == MOE_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = MOE_ERR_CUDA;
      }
      if (rc != MOE_OK) {
        restore();
        return rc;
      }
      for (int k = 0; k < kKinds; ++k) {
        double ms = 0;
        int n = 0;
        moe_trace_read(kTraceOf[k], &ms, &n);
        if (n <= 0) continue;
        const double us = 1000.0 * ms / n;
        if (best[k] < 0 || us < best[k] * (1.0 - kMargin)) {
          best[k] = us;
          out->pair[k] = pair;
          out->prefetch_kb[k] = kDepths[di];
        }
      }
    }
  }
  int mask = 0;
  for (int k = 0; k < kKinds; ++k) {
    if (best[k] < 0) {  // kind never launched: keep the defaults
      out->pair[k] = (prev_mask >> k) & 1;
      out->prefetch_kb[k] = prev_depth[k];
    }
    mask |= out->pair[k] << k;
    out->us[k] = best[k] < 0 ? 0.f : static_cast<float>(best[k]);
    set_gemm_prefetch(static_cast<GemmKind>(k), out->prefetch_kb[k]);
  }
  set_gemm_pair_kinds(mask);
  moe_trace_reset();
  moe_set_bwd_overlap(prev_overlap);
  return MOE_OK;
}

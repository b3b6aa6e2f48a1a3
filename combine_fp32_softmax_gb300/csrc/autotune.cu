// Measured autotuner for the grouped GEMMs and the forward/backward variants:
// per GEMM kind the tile shape (one CTA per 128 x 256 tile, or a CTA pair
// per 256 x 256 tile), the depth of the next-tile L2 prefetch, the tile order
// of the weight-gradient kinds and the pipeline depth, then whether the
// MegaKernels beat the kernel chains, all chosen by timing the caller's own
// layer.  None of these choices changes any arithmetic, so results are the
// same bits before and after tuning.
//
// UniEP page ("Unified Expert-Parallel MoE MegaKernel for LLM Training"),
// section 3 (autotuning, the analytical model and priority scheduling) names
// the step but gives no content; this is the plainest reading: measure the
// candidates on the workload and keep the fastest per kernel.  The search is
// coordinate-wise: each phase fixes the choices of the ones before.
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
// ties keep the first candidate timed: the library's defaults.
constexpr double kMargin = 0.01;

struct Settings {
  int mask;
  int depth[kKinds], order[kKinds], stages[kKinds], epi[kKinds];
};

Settings read_settings() {
  using namespace moe;
  Settings st{};
  st.mask = set_gemm_pair_kinds(0);
  set_gemm_pair_kinds(st.mask);
  for (int k = 0; k < kKinds; ++k) {
    const GemmKind g = static_cast<GemmKind>(k);
    st.depth[k] = set_gemm_prefetch(g, 0);
    set_gemm_prefetch(g, st.depth[k]);
    st.stages[k] = set_gemm_stages(g, 0);
    set_gemm_stages(g, st.stages[k]);
    const int o = set_gemm_tile_order(g, 0);
    st.order[k] = o < 0 ? 0 : o;
    if (o >= 0) set_gemm_tile_order(g, o);
    const int e = set_gemm_epilogue(g, 0);
    st.epi[k] = e < 0 ? 0 : e;
    if (e >= 0) set_gemm_epilogue(g, e);
  }
  return st;
}

void apply_settings(const Settings& st) {
  using namespace moe;
  set_gemm_pair_kinds(st.mask);
  for (int k = 0; k < kKinds; ++k) {
    const GemmKind g = static_cast<GemmKind>(k);
    set_gemm_prefetch(g, st.depth[k]);
    set_gemm_stages(g, st.stages[k]);
    set_gemm_tile_order(g, st.order[k]);  // refused (-1) for the ragged-M kinds
    set_gemm_epilogue(g, st.epi[k]);      // refused for GEMM 1 and dH
  }
}

}  // namespace

extern "C" int moe_autotune(const moe_cfg* cfg, const float* logits, const uint16_t* x, const uint16_t* W1,
                            const uint16_t* W3, const uint16_t* W2, const uint16_t* dy, float* y,
                            int32_t* topk_idx, float* topk_w, float* dx, float* dlogits, float* dW1, float* dW3,
                            float* dW2, void* ws, int reps, void* stream, moe_tune_result* out) {
  using namespace moe;
  if (!out || reps < 0) return MOE_ERR_ARG;
  if (reps == 0) reps = 2;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Settings prev = read_settings();
  // The backward's B/W overlap is off while timing: a weight-gradient GEMM
  // on the second stream would otherwise be charged its wait for the SMs
  // that dX holds.
  const int prev_overlap = moe_set_bwd_overlap(0);
  cudaEvent_t ev0 = nullptr, ev1 = nullptr;
  auto restore = [&](const Settings& st) {
    apply_settings(st);
    moe_trace_enable(0);
    moe_set_bwd_overlap(prev_overlap);
    if (ev0) cudaEventDestroy(ev0);
    if (ev1) cudaEventDestroy(ev1);
  };
  auto fwd = [&](int mk) { return moe_layer_fwd(cfg, logits, x, W1, W3, W2, y, topk_idx, topk_w, ws, mk, stream); };
  auto bwd = [&](int mk) {
    return moe_layer_bwd(cfg, dy, logits, x, W1, W3, W2, topk_idx, topk_w, ws, dx, dlogits, dW1, dW3, dW2,
                         3 | (mk ? MOE_BWD_MEGAKERNEL : 0), stream);
  };
  auto step = [&]() -> int {
    int rc = fwd(0);
    return rc == MOE_OK ? bwd(0) : rc;
  };
  // One candidate: a warm-up step (first launches set attributes and tensor
  // maps), then `reps` steps with per-kernel events; us[k] = microseconds
  // per launch of kind k (-1 when it did not launch).
  auto time_candidate = [&](double* us) -> int {
    moe_trace_enable(0);
    int rc = step();
    if (rc == MOE_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = MOE_ERR_CUDA;
    if (rc != MOE_OK) return rc;
    moe_trace_reset();
    moe_trace_enable(1);
    for (int r = 0; r < reps && rc == MOE_OK; ++r) rc = step();
    moe_trace_enable(0);
    if (rc == MOE_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = MOE_ERR_CUDA;
    for (int k = 0; k < kKinds; ++k) {
      double ms = 0;
      int n = 0;
      moe_trace_read(kTraceOf[k], &ms, &n);
      us[k] = n > 0 ? 1000.0 * ms / n : -1.0;
    }
    return rc;
  };

  Settings cur = prev;
  double best[kKinds];
  for (int k = 0; k < kKinds; ++k) best[k] = -1.0;
  auto keep_if_faster = [&](const double* us, auto&& take) {
    for (int k = 0; k < kKinds; ++k) {
      if (us[k] < 0) continue;
      if (best[k] < 0 || us[k] < best[k] * (1.0 - kMargin)) {
        best[k] = us[k];
        take(k);
      }
    }
  };

  // Phase 1: tile shape x L2 prefetch depth (CTA pairs without prefetch first).
  Settings chosen = cur;
  for (int pi = 0; pi < 2; ++pi) {
    const int pair = 1 - pi;
    for (int di = 0; di < kNumDepths; ++di) {
      Settings c = cur;
      c.mask = pair ? (1 << kKinds) - 1 : 0;
      for (int k = 0; k < kKinds; ++k) c.depth[k] = kDepths[di];
      apply_settings(c);
      double us[kKinds];
      const int rc = time_candidate(us);
      if (rc != MOE_OK) {
        restore(prev);
        return rc;
      }
      keep_if_faster(us, [&](int k) {
        chosen.mask = (chosen.mask & ~(1 << k)) | (pair << k);
        chosen.depth[k] = kDepths[di];
      });
    }
  }
  cur = chosen;
  // Phase 2: the weight-gradient kinds' tile order (long segments' tiles
  // interleaved with the short ones instead of longest first).
  {
    Settings c = cur;
    c.order[kDW13] = c.order[kDW13] ? 0 : 1;
    c.order[kDW2] = c.order[kDW2] ? 0 : 1;
    apply_settings(c);
    double us[kKinds];
    const int rc = time_candidate(us);
    if (rc != MOE_OK) {
      restore(prev);
      return rc;
    }
    us[kG1] = us[kG2] = us[kDH] = us[kDX] = -1.0;  // unchanged kinds: keep their phase-1 times
    keep_if_faster(us, [&](int k) { chosen.order[k] = c.order[k]; });
  }
  cur = chosen;
  // Phase 2b: the fp32-output kinds' epilogue stores (the other mode).
  {
    Settings c = cur;
    for (int k : {static_cast<int>(kG2), static_cast<int>(kDX), static_cast<int>(kDW13), static_cast<int>(kDW2)})
      c.epi[k] = c.epi[k] ? 0 : 1;
    apply_settings(c);
    double us[kKinds];
    const int rc = time_candidate(us);
    if (rc != MOE_OK) {
      restore(prev);
      return rc;
    }
    us[kG1] = us[kDH] = -1.0;
    keep_if_faster(us, [&](int k) { chosen.epi[k] = c.epi[k]; });
  }
  cur = chosen;
  // Phase 3: one pipeline stage fewer than fits (with each kind's epilogue
  // stores; direct stores leave room for one stage more).
  {
    Settings c = cur;
    for (int k = 0; k < kKinds; ++k)
      c.stages[k] = gemm_max_stages(static_cast<GemmKind>(k), ((c.mask >> k) & 1) ? 2 : 1, c.epi[k]) - 1;
    apply_settings(c);
    double us[kKinds];
    const int rc = time_candidate(us);
    if (rc != MOE_OK) {
      restore(prev);
      return rc;
    }
    keep_if_faster(us, [&](int k) { chosen.stages[k] = c.stages[k]; });
  }
  cur = chosen;
  apply_settings(cur);

  // Phase 4: kernel chain against MegaKernel, forward and backward, with the
  // GEMM choices above (a MegaKernel runs its tiles one CTA each).
  if (cudaEventCreate(&ev0) != cudaSuccess || cudaEventCreate(&ev1) != cudaSuccess) {
    restore(prev);
    return MOE_ERR_CUDA;
  }
  float fb_us[2][2] = {{0, 0}, {0, 0}};  // [fwd, bwd][chain, MegaKernel]
  for (int part = 0; part < 2; ++part) {
    for (int mk = 0; mk < 2; ++mk) {
      auto call = [&]() { return part == 0 ? fwd(mk) : bwd(mk); };
      int rc = call();  // warm-up (the backward reads what the last forward left in ws)
      if (rc == MOE_OK) rc = cudaEventRecord(ev0, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
      for (int r = 0; r < reps && rc == MOE_OK; ++r) rc = call();
      if (rc == MOE_OK) rc = cudaEventRecord(ev1, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
      float ms = 0.f;
      if (rc == MOE_OK && (cudaEventSynchronize(ev1) != cudaSuccess || cudaEventElapsedTime(&ms, ev0, ev1) != cudaSuccess))
        rc = MOE_ERR_CUDA;
      if (rc != MOE_OK) {
        restore(prev);
        return rc;
      }
      fb_us[part][mk] = 1000.f * ms / reps;
    }
    if (part == 0 && fwd(0) != MOE_OK) {  // the backward is timed on the chain forward's state
      restore(prev);
      return MOE_ERR_CUDA;
    }
  }
  out->fwd_megakernel = fb_us[0][1] < fb_us[0][0] * (1.0 - kMargin) ? 1 : 0;
  out->bwd_megakernel = fb_us[1][1] < fb_us[1][0] * (1.0 - kMargin) ? 1 : 0;
  for (int v = 0; v < 2; ++v) {
    out->fwd_us[v] = fb_us[0][v];
    out->bwd_us[v] = fb_us[1][v];
  }

  for (int k = 0; k < kKinds; ++k) {
    out->pair[k] = (cur.mask >> k) & 1;
    out->prefetch_kb[k] = cur.depth[k];
    out->tile_order[k] = cur.order[k];
    out->epi_direct[k] = cur.epi[k];
    out->stages[k] = cur.stages[k] > 0 ? cur.stages[k]
                                       : gemm_max_stages(static_cast<GemmKind>(k), out->pair[k] ? 2 : 1, cur.epi[k]);
    out->us[k] = best[k] < 0 ? 0.f : static_cast<float>(best[k]);
  }
  moe_trace_reset();
  moe_set_bwd_overlap(prev_overlap);
  cudaEventDestroy(ev0);
  cudaEventDestroy(ev1);
  return MOE_OK;
}

// C ABI entry points (declared in include/moe.h): argument checks, workspace
// carving and the launch sequences of the forward and backward passes.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"

namespace moe {
int megakernel_fwd(const moe_cfg& c, const WsLayout& L, uint8_t* ws, const uint16_t* x, const uint16_t* W1,
                   const uint16_t* W3, const uint16_t* W2, const float* topk_w, float* y, int grid_limit,
                   cudaStream_t s);
int megakernel_bwd_input(const moe_cfg& c, const WsLayout& L, uint8_t* ws, const GemmArgs& a, const uint16_t* dy,
                         float* dx, int grid, cudaStream_t s);
}

using namespace moe;

namespace {

int g_grid_limit = 0;
int g_route_fusion = 1;
int g_bwd_overlap = 1;
int g_bwd_fused = 0;

// Per device: a second stream and two events for the backward's fork/join
// (weight gradients beside the input-gradient tail).  Created on first use,
// kept until exit.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxDevices = 64;
SideStream g_side[kMaxDevices];
std::mutex g_side_mu;

const SideStream* side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_side_mu);
  SideStream& ss = g_side[dev];
  if (!ss.s) {
    if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess) return ss.s = nullptr, nullptr;
    if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
  }
  return &ss;
}

int persistent_grid() {
  const int n = num_sms();
  return g_grid_limit > 0 ? std::min(g_grid_limit, n) : n;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cfg(const moe_cfg* c) {
  if (!c) return MOE_ERR_ARG;
  if (c->T < 1 || c->d_model < 64 || c->d_ff < 64 || c->E < 1 || c->k < 1 || c->n_shared < 0) return MOE_ERR_SHAPE;
  if (c->E > 256 || c->k > c->E || c->k > 8 || c->n_shared > 4) return MOE_ERR_SHAPE;
  if (c->d_model % 64 || c->d_ff % 64) return MOE_ERR_SHAPE;
  if (c->renorm != 0 && c->renorm != 1) return MOE_ERR_SHAPE;
  if (static_cast<long long>(c->T) * (c->k + c->n_shared) >= (1ll << 31) - 256) return MOE_ERR_SHAPE;
  return MOE_OK;
}

// Checks required (non-null, 16-byte aligned) and optional (aligned if set)
// pointers plus the workspace.
int check_ptrs(std::initializer_list<const void*> req, std::initializer_list<const void*> opt, const void* ws) {
  for (const void* p : req) {
    if (!p) return MOE_ERR_ARG;
    if (!al16(p)) return MOE_ERR_ALIGN;
  }
  for (const void* p : opt)
    if (p && !al16(p)) return MOE_ERR_ALIGN;
  if (!ws) return MOE_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_ALIGN;
  return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)             \
  do {                            \
    const int _rc = (expr);       \
    if (_rc != MOE_OK) return _rc; \
  } while (0)
#define MOE_TRY_CUDA(expr) MOE_TRY(cuda_status(expr))

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

GemmArgs base_args(const moe_cfg& c, void* ws, const WsLayout& L) {
  GemmArgs a{};
  a.T = c.T;
  a.d = c.d_model;
  a.f = c.d_ff;
  a.E = c.E;
  a.k = c.k;
  a.S = c.n_shared;
  a.err = at<int>(ws, L.err);
  return a;
}

// Permutation builder from a histogram already in ws.hist.
int build_tables(const moe_cfg& c, const WsLayout& L, void* ws, const int32_t* topk_idx, int32_t* counts,
                 int32_t* offsets, int32_t* dest, int32_t* row_token, int32_t* row_slot, cudaStream_t s) {
  const int R = c.T * c.k;
  MOE_TRY_CUDA(launch_scan(at<int32_t>(ws, L.hist), c.E, L.nb_route, R, at<int32_t>(ws, L.base), counts, offsets, s));
  MOE_TRY_CUDA(launch_scatter(topk_idx, at<int32_t>(ws, L.base), c.T, c.E, c.k, L.nb_route, dest, row_token,
                              row_slot, at<int>(ws, L.err), s));
  return MOE_OK;
}

// Router and permutation tables of the layer forward: one cooperative
// launch, else (fusion off or refused) the router and build_tables.
int route_tables(const moe_cfg& c, const WsLayout& L, void* ws, const float* logits, int32_t* topk_idx,
                 float* topk_w, cudaStream_t s) {
  int32_t* hist = at<int32_t>(ws, L.hist);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* dest = at<int32_t>(ws, L.dest);
  int32_t* row_token = at<int32_t>(ws, L.row_token);
  int32_t* row_slot = at<int32_t>(ws, L.row_slot);
  int* err = at<int>(ws, L.err);
  if (g_route_fusion) {
    const cudaError_t e =
        launch_route_tables(logits, c.T, c.E, c.k, c.renorm, L.nb_route, topk_idx, topk_w, hist,
                            at<int32_t>(ws, L.base), counts, offsets, dest, row_token, row_slot, err,
                            g_grid_limit, s);
    if (e == cudaSuccess) return MOE_OK;
    if (e != cudaErrorCooperativeLaunchTooLarge && e != cudaErrorNotSupported) return MOE_ERR_CUDA;
    (void)cudaGetLastError();  // not a sticky error: take the three-kernel path
  }
  MOE_TRY_CUDA(launch_route(logits, c.T, c.E, c.k, c.renorm, topk_idx, topk_w, hist, L.nb_route, err, s));
  return build_tables(c, L, ws, topk_idx, counts, offsets, dest, row_token, row_slot, s);
}

int fwd_gemms(const moe_cfg& c, const WsLayout& L, void* ws, const uint16_t* Xp, const uint16_t* x,
              const int32_t* offsets, const int32_t* row_slot, const float* topk_w, const uint16_t* W1,
              const uint16_t* W3, const uint16_t* W2, uint16_t* Hw, uint16_t* AB, float* Op, cudaStream_t s) {
  GemmArgs a = base_args(c, ws, L);
  a.offsets = offsets;
  a.row_slot = row_slot;
  a.topk_w = topk_w;
  a.Xp = Xp;
  a.x = x;
  a.W1 = W1;
  a.W3 = W3;
  a.W2 = W2;
  a.Hw = Hw;
  a.Hw_out = Hw;
  a.AB_out = AB;
  a.Op_out = Op;
  MOE_TRY(launch_gemm(kG1, a, s, persistent_grid()));
  MOE_TRY(launch_gemm(kG2, a, s, persistent_grid()));
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const moe_cfg* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return ws_layout(*cfg).total;
}

int moe_ws_init(const moe_cfg* cfg, void* ws, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_ptrs({}, {}, ws));
  const WsLayout L = ws_layout(*cfg);
  MOE_TRY_CUDA(cudaMemsetAsync(at<uint8_t>(ws, L.err), 0, kErrRegionBytes, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_num_sms(void) { return num_sms(); }

int moe_set_grid_limit(int n) {
  g_grid_limit = n > 0 ? n : 0;
  return MOE_OK;
}

int moe_set_gemm_pair_kinds(int mask) { return set_gemm_pair_kinds(mask); }

int moe_set_route_fusion(int on) {
  const int prev = g_route_fusion;
  g_route_fusion = on != 0;
  return prev;
}

int moe_set_bwd_fused_gemms(int on) {
  const int prev = g_bwd_fused;
  g_bwd_fused = on != 0;
  return prev;
}

int moe_set_bwd_overlap(int on) {
  const int prev = g_bwd_overlap;
  g_bwd_overlap = on != 0;
  return prev;
}

int moe_set_gemm_prefetch(int kind, int kblocks) {
  if (kind < kG1 || kind > kDW2) return MOE_ERR_ARG;
  return set_gemm_prefetch(static_cast<GemmKind>(kind), kblocks);
}

int moe_set_gemm_tile_order(int kind, int order) {
  if (kind != kDW13 && kind != kDW2) return MOE_ERR_ARG;
  if (order != 0 && order != 1) return MOE_ERR_ARG;
  return set_gemm_tile_order(static_cast<GemmKind>(kind), order);
}

int moe_set_gemm_epilogue(int kind, int direct) {
  if ((kind != kG2 && kind != kDX && kind != kDW13 && kind != kDW2) || (direct != 0 && direct != 1))
    return MOE_ERR_ARG;
  return set_gemm_epilogue(static_cast<GemmKind>(kind), direct);
}

int moe_set_gemm_stages(int kind, int stages) {
  if (kind < kG1 || kind > kDW2 || stages < 0) return MOE_ERR_ARG;
  return set_gemm_stages(static_cast<GemmKind>(kind), stages);
}

int moe_gemm_max_stages(int kind, int cta_group) {
  if (kind < kG1 || kind > kDW2 || (cta_group != 1 && cta_group != 2)) return 0;
  return gemm_max_stages(static_cast<GemmKind>(kind), cta_group);
}

int moe_gemm_pair_capacity(int kind) {
  if (kind < kG1 || kind > kDW2) return 0;
  return gemm_pair_capacity(static_cast<GemmKind>(kind));
}

int moe_route(const moe_cfg* cfg, const float* logits, int32_t* topk_idx, float* topk_w, void* ws, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_ptrs({logits, topk_idx, topk_w}, {}, ws));
  const WsLayout L = ws_layout(*cfg);
  const moe_cfg& c = *cfg;
  MOE_TRY_CUDA(launch_route(logits, c.T, c.E, c.k, c.renorm, topk_idx, topk_w, at<int32_t>(ws, L.hist), L.nb_route,
                            at<int>(ws, L.err), static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_dispatch(const moe_cfg* cfg, const int32_t* topk_idx, const uint16_t* x, int32_t* counts, int32_t* offsets,
                 int32_t* dest, int32_t* row_token, int32_t* row_slot, uint16_t* Xp, void* ws, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_ptrs({topk_idx, counts, offsets, dest, row_token, row_slot}, {x, Xp}, ws));
  const WsLayout L = ws_layout(*cfg);
  const moe_cfg& c = *cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_TRY_CUDA(launch_hist(topk_idx, c.T, c.E, c.k, at<int32_t>(ws, L.hist), L.nb_route, at<int>(ws, L.err), s));
  MOE_TRY(build_tables(c, L, ws, topk_idx, counts, offsets, dest, row_token, row_slot, s));
  if (x && Xp) MOE_TRY_CUDA(launch_scatter_rows_bf16(x, dest, c.T, c.k, c.d_model, Xp, MOE_K_GATHER, at<int>(ws, L.err), s));
  return MOE_OK;
}

int moe_token_addresses(const moe_cfg* cfg, const int32_t* topk_idx, const int32_t* rank_base, int32_t* counts,
                        int32_t* offsets, int32_t* dest, void* ws, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_ptrs({topk_idx, counts, offsets, dest}, {rank_base}, ws));
  const WsLayout L = ws_layout(*cfg);
  const moe_cfg& c = *cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* base = at<int32_t>(ws, L.base);
  MOE_TRY_CUDA(launch_hist(topk_idx, c.T, c.E, c.k, at<int32_t>(ws, L.hist), L.nb_route, at<int>(ws, L.err), s));
  MOE_TRY_CUDA(launch_scan(at<int32_t>(ws, L.hist), c.E, L.nb_route, c.T * c.k, base, counts, offsets, s));
  if (rank_base) MOE_TRY_CUDA(launch_rebase(base, offsets, rank_base, c.E, L.nb_route, s));
  MOE_TRY_CUDA(launch_scatter(topk_idx, base, c.T, c.E, c.k, L.nb_route, dest, nullptr, nullptr, at<int>(ws, L.err), s));
  return MOE_OK;
}

int moe_rank_bases(const int32_t* all_counts, int G, int E, const int32_t* owner, int rank, int32_t* rank_base,
                   int32_t* recv_rows, void* stream) {
  if (G < 1 || G > 65536 || E < 1 || E > 256 || rank < 0 || rank >= G) return MOE_ERR_SHAPE;
  if (!all_counts || !owner || !rank_base) return MOE_ERR_ARG;
  if (!al16(all_counts) || !al16(owner) || !al16(rank_base) || (recv_rows && !al16(recv_rows))) return MOE_ERR_ALIGN;
  MOE_TRY_CUDA(launch_rank_bases(all_counts, G, E, owner, rank, rank_base, recv_rows,
                                 static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_group_gemm_swiglu(const moe_cfg* cfg, const uint16_t* Xp, const uint16_t* x, const int32_t* offsets,
                          const int32_t* row_slot, const float* topk_w, const uint16_t* W1, const uint16_t* W3,
                          const uint16_t* W2, uint16_t* Hw, uint16_t* AB, float* Oprime, void* ws, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_ptrs({Xp, offsets, row_slot, topk_w, W1, W3, W2, Hw, Oprime}, {x, AB}, ws));
  if (cfg->n_shared > 0 && !x) return MOE_ERR_ARG;
  const WsLayout L = ws_layout(*cfg);
  return fwd_gemms(*cfg, L, ws, Xp, x, offsets, row_slot, topk_w, W1, W3, W2, Hw, AB, Oprime,
                   static_cast<cudaStream_t>(stream));
}

int moe_combine(const moe_cfg* cfg, const float* Oprime, const int32_t* dest, float* y, void* ws, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_ptrs({Oprime, dest, y}, {}, ws));
  const moe_cfg& c = *cfg;
  MOE_TRY_CUDA(launch_sum_rows_f32(Oprime, dest, c.T, c.k, c.n_shared, c.d_model, y, MOE_K_COMBINE, at<int>(ws, 0), static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_layer_fwd(const moe_cfg* cfg, const float* logits, const uint16_t* x, const uint16_t* W1, const uint16_t* W3,
                  const uint16_t* W2, float* y, int32_t* topk_idx, float* topk_w, void* ws, int use_megakernel,
                  void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_ptrs({logits, x, W1, W3, W2, y, topk_idx, topk_w}, {}, ws));
  const moe_cfg& c = *cfg;
  const WsLayout L = ws_layout(c);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int R = c.T * c.k;
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* row_token = at<int32_t>(ws, L.row_token);
  int32_t* row_slot = at<int32_t>(ws, L.row_slot);
  int32_t* dest = at<int32_t>(ws, L.dest);
  MOE_TRY(route_tables(c, L, ws, logits, topk_idx, topk_w, s));
  if (use_megakernel)
    return megakernel_fwd(c, L, static_cast<uint8_t*>(ws), x, W1, W3, W2, topk_w, y, persistent_grid(), s);
  uint16_t* Xp = at<uint16_t>(ws, L.Xp);
  float* Op = at<float>(ws, L.Op);
  MOE_TRY_CUDA(launch_scatter_rows_bf16(x, dest, c.T, c.k, c.d_model, Xp, MOE_K_GATHER, at<int>(ws, L.err), s));
  MOE_TRY(fwd_gemms(c, L, ws, Xp, x, offsets, row_slot, topk_w, W1, W3, W2, at<uint16_t>(ws, L.Hw),
                    at<uint16_t>(ws, L.AB), Op, s));
  MOE_TRY_CUDA(launch_sum_rows_f32(Op, dest, c.T, c.k, c.n_shared, c.d_model, y, MOE_K_COMBINE, at<int>(ws, L.err), s));
  return MOE_OK;
}

int moe_combine_bwd(const moe_cfg* cfg, const uint16_t* dy, const int32_t* row_token, uint16_t* G, void* ws,
                    void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_ptrs({dy, row_token, G}, {}, ws));
  const moe_cfg& c = *cfg;
  MOE_TRY_CUDA(launch_gather_rows_bf16(dy, row_token, c.T, c.T * c.k, c.d_model, G, MOE_K_COMBINE_BWD, at<int>(ws, 0), static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_group_gemm_swiglu_bwd(const moe_cfg* cfg, const uint16_t* G, const uint16_t* dy, const uint16_t* Xp,
                              const uint16_t* x, const int32_t* offsets, const int32_t* row_slot, const int32_t* dest,
                              const float* topk_w, const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                              const uint16_t* Hw, const uint16_t* AB, uint16_t* dAB, float* dw,
                              float* dXp, float* dW1, float* dW3, float* dW2, int which, void* ws, void* stream) {
  MOE_TRY(check_cfg(cfg));
  if (which < 1 || which > 3) return MOE_ERR_ARG;
  MOE_TRY(check_ptrs({G, dy, offsets, row_slot, dAB}, {Xp, x, dest, topk_w, W1, W3, W2, Hw, AB, dw, dXp, dW1, dW3, dW2}, ws));
  if ((which & 1) && !(dest && topk_w && W1 && W3 && W2 && AB && dw && dXp)) return MOE_ERR_ARG;
  if ((which & 2) && !(Xp && Hw && dW1 && dW3 && dW2)) return MOE_ERR_ARG;
  if (cfg->n_shared > 0 && (which & 2) && !x) return MOE_ERR_ARG;
  const moe_cfg& c = *cfg;
  const WsLayout L = ws_layout(c);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemmArgs a = base_args(c, ws, L);
  a.offsets = offsets;
  a.row_slot = row_slot;
  a.topk_w = topk_w;
  a.Xp = Xp;
  a.x = x;
  a.W1 = W1;
  a.W3 = W3;
  a.W2 = W2;
  a.AB = AB;
  a.G = G;
  a.dy = dy;
  a.dAB = dAB;
  a.Hw = Hw;
  a.dAB_out = dAB;
  a.partial_out = at<float>(ws, L.partial);
  a.dXp_out = dXp;
  a.dW1_out = dW1;
  a.dW3_out = dW3;
  a.dW2_out = dW2;
  if (which & 1) {
    MOE_TRY(launch_gemm(kDH, a, s, persistent_grid()));
    MOE_TRY_CUDA(launch_dw_reduce(a.partial_out, dest, c.T * c.k, L.nt_dh, dw, at<int>(ws, L.err), s));
    MOE_TRY(launch_gemm(kDX, a, s, persistent_grid()));
  }
  if (which & 2) {
    MOE_TRY(launch_gemm(kDW13, a, s, persistent_grid()));
    MOE_TRY(launch_gemm(kDW2, a, s, persistent_grid()));
  }
  return MOE_OK;
}

int moe_dispatch_bwd(const moe_cfg* cfg, const float* dXp, const int32_t* dest, float* dx, void* ws, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_ptrs({dXp, dest, dx}, {}, ws));
  const moe_cfg& c = *cfg;
  MOE_TRY_CUDA(launch_sum_rows_f32(dXp, dest, c.T, c.k, c.n_shared, c.d_model, dx, MOE_K_DISPATCH_BWD, at<int>(ws, 0), static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_route_bwd(const moe_cfg* cfg, const float* logits, const int32_t* topk_idx, const float* topk_w,
                  const float* dw, float* dlogits, void* ws, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_ptrs({logits, topk_idx, topk_w, dw, dlogits}, {}, ws));
  const moe_cfg& c = *cfg;
  MOE_TRY_CUDA(launch_route_bwd(logits, topk_idx, topk_w, dw, c.T, c.E, c.k, c.renorm, dlogits, at<int>(ws, 0),
                                static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_layer_bwd(const moe_cfg* cfg, const uint16_t* dy, const float* logits, const uint16_t* x, const uint16_t* W1,
                  const uint16_t* W3, const uint16_t* W2, const int32_t* topk_idx, const float* topk_w, void* ws,
                  float* dx, float* dlogits, float* dW1, float* dW3, float* dW2, int which, void* stream) {
  MOE_TRY(check_cfg(cfg));
  const bool mega = (which & MOE_BWD_MEGAKERNEL) != 0;
  which &= ~MOE_BWD_MEGAKERNEL;
  if (which < 1 || which > 3) return MOE_ERR_ARG;
  MOE_TRY(check_ptrs({dy, logits, x, W1, W3, W2, topk_idx, topk_w}, {dx, dlogits, dW1, dW3, dW2}, ws));
  if ((which & 1) && !(dx && dlogits)) return MOE_ERR_ARG;
  if ((which & 2) && !(dW1 && dW3 && dW2)) return MOE_ERR_ARG;
  const moe_cfg& c = *cfg;
  const WsLayout L = ws_layout(c);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int R = c.T * c.k;
  const int32_t* offsets = at<int32_t>(ws, L.offsets);
  const int32_t* row_token = at<int32_t>(ws, L.row_token);
  const int32_t* row_slot = at<int32_t>(ws, L.row_slot);
  const int32_t* dest = at<int32_t>(ws, L.dest);
  uint16_t* G = at<uint16_t>(ws, L.G);
  uint16_t* dAB = at<uint16_t>(ws, L.dAB);
  const uint16_t* Hw = at<uint16_t>(ws, L.Hw);
  float* dXp = at<float>(ws, L.dXp);
  float* dw = at<float>(ws, L.dw);
  GemmArgs a = base_args(c, ws, L);
  a.offsets = offsets;
  a.row_slot = row_slot;
  a.topk_w = topk_w;
  a.Xp = at<uint16_t>(ws, L.Xp);
  a.x = x;
  a.W1 = W1;
  a.W3 = W3;
  a.W2 = W2;
  a.AB = at<uint16_t>(ws, L.AB);
  a.G = G;
  a.dy = dy;
  a.dAB = dAB;
  a.Hw = Hw;
  a.dAB_out = dAB;
  a.partial_out = at<float>(ws, L.partial);
  a.dXp_out = dXp;
  a.dW1_out = dW1;
  a.dW3_out = dW3;
  a.dW2_out = dW2;
  // B/W split (GraphPP page, section 2: the backward splits into its
  // input-gradient part B and its deferrable weight-gradient part W): the W
  // GEMMs need only dH's outputs, so with which == 3 they run on a second
  // stream forked after dH and fill the SMs that dX's tail frees and that
  // the memory-bound dx sum and router backward leave idle.  The streams
  // join before return; no arithmetic moves, so the bits are unchanged.
  const SideStream* side = (which == 3 && g_bwd_overlap) ? side_stream() : nullptr;
  if (which == 3 && g_bwd_overlap && !side) return MOE_ERR_CUDA;
  if ((which & 1) && mega) {  // B part as one MegaKernel, then the two small router-gradient launches
    MOE_TRY(megakernel_bwd_input(c, L, static_cast<uint8_t*>(ws), a, dy, dx, persistent_grid(), s));
    if (side) {  // the W GEMMs beside the dw reduce and router backward
      MOE_TRY_CUDA(cudaEventRecord(side->fork, s));
      MOE_TRY_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
      MOE_TRY(launch_gemm(kDW13, a, side->s, persistent_grid()));
      MOE_TRY(launch_gemm(kDW2, a, side->s, persistent_grid()));
      MOE_TRY_CUDA(cudaEventRecord(side->join, side->s));
    }
    MOE_TRY_CUDA(launch_dw_reduce(a.partial_out, dest, R, L.nt_dh, dw, at<int>(ws, L.err), s));
    MOE_TRY_CUDA(launch_route_bwd(logits, topk_idx, topk_w, dw, c.T, c.E, c.k, c.renorm, dlogits, at<int>(ws, L.err), s));
    if (side) {
      MOE_TRY_CUDA(cudaStreamWaitEvent(s, side->join, 0));
      return MOE_OK;
    }
  } else if (which == 3 && g_bwd_fused) {  // dX and the W GEMMs interleaved in one launch
    MOE_TRY_CUDA(launch_scatter_rows_bf16(dy, dest, c.T, c.k, c.d_model, G, MOE_K_COMBINE_BWD, at<int>(ws, L.err), s));
    MOE_TRY(launch_gemm(kDH, a, s, persistent_grid()));
    MOE_TRY_CUDA(launch_dw_reduce(a.partial_out, dest, R, L.nt_dh, dw, at<int>(ws, L.err), s));
    MOE_TRY_CUDA(launch_route_bwd(logits, topk_idx, topk_w, dw, c.T, c.E, c.k, c.renorm, dlogits, at<int>(ws, L.err), s));
    MOE_TRY(launch_bwd_gemms(a, s, persistent_grid()));
    MOE_TRY_CUDA(launch_sum_rows_f32(dXp, dest, c.T, c.k, c.n_shared, c.d_model, dx, MOE_K_DISPATCH_BWD, at<int>(ws, L.err), s));
    return MOE_OK;
  } else if (which & 1) {  // B part: input gradients (critical path)
    MOE_TRY_CUDA(launch_scatter_rows_bf16(dy, dest, c.T, c.k, c.d_model, G, MOE_K_COMBINE_BWD, at<int>(ws, L.err), s));
    MOE_TRY(launch_gemm(kDH, a, s, persistent_grid()));
    if (side) {
      MOE_TRY_CUDA(cudaEventRecord(side->fork, s));
      MOE_TRY(launch_gemm(kDX, a, s, persistent_grid()));  // queued first: it has the SMs first
      MOE_TRY_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
      MOE_TRY(launch_gemm(kDW13, a, side->s, persistent_grid()));
      MOE_TRY(launch_gemm(kDW2, a, side->s, persistent_grid()));
      MOE_TRY_CUDA(cudaEventRecord(side->join, side->s));
      MOE_TRY_CUDA(launch_dw_reduce(a.partial_out, dest, R, L.nt_dh, dw, at<int>(ws, L.err), s));
      MOE_TRY_CUDA(launch_route_bwd(logits, topk_idx, topk_w, dw, c.T, c.E, c.k, c.renorm, dlogits, at<int>(ws, L.err), s));
      MOE_TRY_CUDA(
          launch_sum_rows_f32(dXp, dest, c.T, c.k, c.n_shared, c.d_model, dx, MOE_K_DISPATCH_BWD, at<int>(ws, L.err), s));
      MOE_TRY_CUDA(cudaStreamWaitEvent(s, side->join, 0));
      return MOE_OK;
    }
    MOE_TRY_CUDA(launch_dw_reduce(a.partial_out, dest, R, L.nt_dh, dw, at<int>(ws, L.err), s));
    MOE_TRY_CUDA(launch_route_bwd(logits, topk_idx, topk_w, dw, c.T, c.E, c.k, c.renorm, dlogits, at<int>(ws, L.err), s));
    MOE_TRY(launch_gemm(kDX, a, s, persistent_grid()));
    MOE_TRY_CUDA(launch_sum_rows_f32(dXp, dest, c.T, c.k, c.n_shared, c.d_model, dx, MOE_K_DISPATCH_BWD, at<int>(ws, L.err), s));
  }
  if (which & 2) {  // W part: weight gradients (deferrable)
    MOE_TRY(launch_gemm(kDW13, a, s, persistent_grid()));
    MOE_TRY(launch_gemm(kDW2, a, s, persistent_grid()));
  }
  return MOE_OK;
}

int moe_get_device_error(const void* ws, void* stream, int* code, int* info) {
  if (!ws || !code || !info) return MOE_ERR_ARG;
  int host[2] = {0, 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The error word is the first field of every workspace layout.
  MOE_TRY_CUDA(cudaMemcpyAsync(host, ws, sizeof(host), cudaMemcpyDeviceToHost, s));
  MOE_TRY_CUDA(cudaStreamSynchronize(s));
  *code = host[0];
  *info = host[1];
  return MOE_OK;
}

}  // extern "C"

// Host-side launchers of the library's kernels (internal; the public entry
// points in api.cu validate arguments and call these).  All launch on
// `stream` and return cudaGetLastError() of the launch.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"

namespace moe {

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* topk_idx,
                         float* topk_w, int32_t* hist, int nb, int* err, cudaStream_t s);
// Router + histogram + scan + stable scatter in one cooperative launch of
// at most max_grid blocks (0: as many as fit).  Returns the launch's error
// without recording it if the device cannot run the grid cooperatively.
cudaError_t launch_route_tables(const float* logits, int T, int E, int k, int renorm, int nb, int32_t* topk_idx,
                                float* topk_w, int32_t* hist, int32_t* base, int32_t* counts, int32_t* offsets,
                                int32_t* dest, int32_t* row_token, int32_t* row_slot, int* err, int max_grid,
                                cudaStream_t s);
cudaError_t launch_hist(const int32_t* topk_idx, int T, int E, int k, int32_t* hist, int nb, int* err,
                        cudaStream_t s);
cudaError_t launch_scan(const int32_t* hist, int E, int nb, int R, int32_t* base, int32_t* counts,
                        int32_t* offsets, cudaStream_t s);
cudaError_t launch_scatter(const int32_t* topk_idx, const int32_t* base, int T, int E, int k, int nb,
                           int32_t* dest, int32_t* row_token, int32_t* row_slot, int* err, cudaStream_t s);
// base[e*nb + b] += rank_base[e] - offsets[e] (multi-rank token mapping).
cudaError_t launch_rebase(int32_t* base, const int32_t* offsets, const int32_t* rank_base, int E, int nb,
                          cudaStream_t s);
// rank_base[e] (and recv_rows[o], if non-null) of the multi-rank token
// mapping from the all-gathered counts [G][E] and the expert owners [E].
cudaError_t launch_rank_bases(const int32_t* counts, int G, int E, const int32_t* owner, int rank,
                              int32_t* rank_base, int32_t* recv_rows, cudaStream_t s);
// dst[r] = src[idx[r]] for r < nrows, rows of `d` bf16 (zero row if the
// index is outside [0, nsrc)).
cudaError_t launch_gather_rows_bf16(const uint16_t* src, const int32_t* idx, int nsrc, int nrows, int d,
                                    uint16_t* dst, int trace_kind, int* err, cudaStream_t s);
// dst[dest[t*k+j]] = src[t] for t < T, j < k (rows of `d` bf16): the rows a
// gather by row_token writes, each source row read once.
cudaError_t launch_scatter_rows_bf16(const uint16_t* src, const int32_t* dest, int T, int k, int d, uint16_t* dst,
                                     int trace_kind, int* err, cudaStream_t s);
// out[t] = sum_j rows[sel[t*k+j]] (slot order) + sum_s rows[R + s*T + t], fp32.
cudaError_t launch_sum_rows_f32(const float* rows, const int32_t* sel, int T, int k, int S, int d, float* out,
                                int trace_kind, int* err, cudaStream_t s);
// dw[i] = sum_nt partial[dest[i] * nt + n] for the T*k slots.
cudaError_t launch_dw_reduce(const float* partial, const int32_t* dest, int R, int nt, float* dw, int* err,
                             cudaStream_t s);
cudaError_t launch_route_bwd(const float* logits, const int32_t* topk_idx, const float* topk_w, const float* dw,
                             int T, int E, int k, int renorm, float* dlogits, int* err, cudaStream_t s);
int num_sms();
// Makes sure the modules of moe_dispatch's kernels (histogram, scan, scatter,
// row gather) are loaded on the current device.
cudaError_t preload_dispatch_kernels();

}  // namespace moe

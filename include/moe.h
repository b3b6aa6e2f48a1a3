/*
 * moe.h — C ABI of libmoe_gb300: the single-GPU hot path of a
 * Mixture-of-Experts layer on GB300 (sm_103a).
 *
 * The layer is the one UniEP fuses into a MegaKernel (UniEP page, "Unified
 * Expert-Parallel MoE MegaKernel for LLM Training", section 1.1, Figure 1):
 *   gate (softmax) -> top-k -> dispatch (scatter) -> GroupGEMM -> SwiGLU ->
 *   GroupGEMM -> combine (weighted sum by gate score),
 * and its backward, which mirrors the forward and needs the transposed
 * GroupGEMM for the weight gradients (same section).  The SwiGLU expert is
 * the MLP of the GraphPP page, sections 5.1-5.2 (gate projection W1, up
 * projection W3, SiLU, gate product, down projection W2).
 *
 * Conventions shared by every call:
 *  - Every data pointer is DEVICE memory owned by the caller.  The library
 *    never allocates, frees or synchronises the host; every call enqueues
 *    work on `stream` (a cudaStream_t passed as void*; NULL = legacy stream)
 *    and returns immediately.
 *  - bf16 tensors are passed as uint16_t* (raw bf16 bit patterns).
 *  - Layouts are row-major.  Weights use the [out, in] layout of a linear
 *    layer: W1, W3 are [E+S, f, d], W2 is [E+S, d, f]; the S shared
 *    experts' weights follow the E routed experts' in the same arrays.
 *  - Row space of the expert GEMMs ("GEMM rows"): rows [0, R) are the R=T*k
 *    routed rows grouped by expert (expert e owns [offsets[e],
 *    offsets[e+1])), rows [R + s*T, R + (s+1)*T) are shared expert s in
 *    token order.  R_s = R + S*T.
 *  - Every pointer must be 16-byte aligned (MOE_ERR_ALIGN otherwise); `ws`
 *    must be 256-byte aligned and at least moe_workspace_bytes() long.
 *  - Return value: MOE_OK, or a negative MOE_ERR_* detected on the host
 *    before anything was enqueued.  Errors found by the kernels themselves
 *    (non-finite logits, a bounded wait that ran out) are recorded in a
 *    device error word inside `ws`; read it with moe_get_device_error().
 *  - Results are bitwise deterministic: no call accumulates floating-point
 *    values with atomics, and every reduction runs in a fixed order.
 *  - Every output is fully overwritten (no accumulate-into mode).
 *  - The layer calls can be captured in a CUDA graph and replayed (stream
 *    capture of the caller's stream, relaxed or thread-local mode): every
 *    launch is capturable, including the cooperative routing launch, the
 *    CTA-pair cluster launches and the fork/join of the backward's second
 *    stream, and the scheduling counters in `ws` reset themselves on the
 *    device.  The first call with a configuration should run uncaptured
 *    (it sets kernel attributes and caches occupancy); moe_autotune and the
 *    moe_trace_* timing calls synchronise and must stay outside a capture.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Layer shape.  T tokens, model width d_model, expert hidden width d_ff,
 * E routed experts, top-k routing, n_shared always-on shared experts,
 * renorm = 0: routing weight = softmax probability of the expert;
 * renorm = 1: probabilities renormalised over the k picks.
 * Limits (MOE_ERR_SHAPE otherwise): 1 <= E <= 256, 1 <= k <= min(E, 8),
 * 0 <= n_shared <= 4, d_model and d_ff multiples of 64, T >= 1,
 * T * (k + n_shared) < 2^31 - 256, renorm in {0, 1}. */
typedef struct moe_cfg {
  int T, d_model, d_ff, E, k, n_shared, renorm;
} moe_cfg;

enum {
  MOE_OK = 0,
  MOE_ERR_ARG = -1,       /* null pointer where one is required */
  MOE_ERR_SHAPE = -2,     /* cfg outside the limits above */
  MOE_ERR_ALIGN = -3,     /* pointer not 16-byte aligned (ws: 256-byte) */
  MOE_ERR_CUDA = -4,      /* a CUDA runtime/driver call or launch failed */
  MOE_ERR_NONFINITE = -5, /* device: a router logit was NaN or Inf */
  MOE_ERR_TIMEOUT = -6    /* device: a bounded wait ran out */
};

/* Bytes of workspace for `cfg`.  The workspace holds the routing tables,
 * the activations the backward needs (Xp, [a|b], Hw, O'), the backward's
 * intermediates, scratch counters and the device error word.  The caller
 * allocates it once; moe_layer_fwd fills it and moe_layer_bwd reads it, so
 * it must stay alive and unmodified between the two.  Calls that share a
 * workspace must not run concurrently on the GPU (e.g. on two streams with
 * no ordering between them): they share its scratch, its scheduling
 * counters and its error word.  Different workspaces are independent. */
size_t moe_workspace_bytes(const moe_cfg* cfg);

/* Clears the device error word in `ws` (async on `stream`).  Call once after
 * allocating the workspace; the layer calls do not clear it. */
int moe_ws_init(const moe_cfg* cfg, void* ws, void* stream);

/* Router (UniEP page, section 1.1: gating probabilities, then top-k).
 * logits [T, E] fp32.  p = softmax over all E (fp32: max-subtract, expf,
 * sum, divide).  The k experts are picked on the LOGITS, larger first, ties
 * to the lower index, -0.0 == +0.0; slot j holds the j-th pick.
 * topk_idx [T, k] int32, topk_w [T, k] fp32 (p, or p / sum of the k picked
 * p when renorm = 1).  A NaN/Inf logit sets MOE_ERR_NONFINITE in the device
 * error word (that token's outputs are then unspecified). */
int moe_route(const moe_cfg* cfg, const float* logits, int32_t* topk_idx,
              float* topk_w, void* ws, void* stream);

/* Deterministic token mapping (UniEP page, section 2.2, Algorithm 1, for a
 * single rank: the cross-rank base offset is 0) and dispatch gather.
 * counts [E]: slots routed to each expert; offsets [E+1]: exclusive prefix
 * sum (offsets[E] = R); dest [R]: flat slot t*k+j -> GEMM row; row_token [R]
 * and row_slot [R]: GEMM row -> token and flat slot.  Within an expert the
 * rows are in ascending flat-slot order, independent of thread scheduling.
 * If x [T, d] (bf16) and Xp [R, d] (bf16) are both non-NULL, also gathers
 * Xp[r] = x[row_token[r]]. */
int moe_dispatch(const moe_cfg* cfg, const int32_t* topk_idx, const uint16_t* x,
                 int32_t* counts, int32_t* offsets, int32_t* dest,
                 int32_t* row_token, int32_t* row_slot, uint16_t* Xp,
                 void* ws, void* stream);

/* moe_dispatch for callers that cannot provide a workspace (no counterpart
 * on the pages: a deployment variant of moe_dispatch).  Some callers may not
 * allocate device memory while they run -- e.g. a framework operator
 * registered with a zero-byte workspace, or code whose device memory a host
 * framework planned in advance -- so they cannot give the library `ws`.
 * This entry point computes exactly what moe_dispatch computes (same
 * arguments minus ws; Xp gathered when x and Xp are both non-NULL), but
 * keeps its scratch (expert histogram, block bases, error word) in a 4 MiB
 * array inside the library, held by every GPU that loads it until exit.
 * After its first call on a device (below) it allocates nothing and calls
 * no allocating routine.
 *  - Limit: E * ceil(T / 32) <= 524,256 (e.g. 64 experts and 262,144
 *    tokens); larger shapes return MOE_ERR_SHAPE before any work.
 *  - The first call on a device sets up (with that device current): it
 *    loads this library's dispatch kernels and the array if the CUDA
 *    runtime has not loaded them yet (under lazy module loading that is
 *    when the 4 MiB array is placed in device memory, an allocation made by
 *    the driver) and looks up the array's device address.  Make that first
 *    call before any stream capture and before any stretch of code in which
 *    nothing may allocate; every later call on that device allocates
 *    nothing.  The set-up is thread-safe; after a device reset the process
 *    must restart before calling this again on that device.
 *  - Every call shares the one array, which keeps the last call's contents:
 *    two calls whose work can overlap on the GPU (e.g. issued on different
 *    streams with no ordering between them) race and produce wrong tables;
 *    order them on one stream or with events.
 *  - Out-of-range expert indices are clamped as in moe_dispatch (the tables
 *    are the ones moe_dispatch gives for the same indices); the call still
 *    returns MOE_OK, and the error record stays inside the array (there is
 *    no workspace to read it from): validate indices beforehand, or use
 *    moe_dispatch and moe_get_device_error, where that matters. */
int moe_dispatch_noalloc(const moe_cfg* cfg, const int32_t* topk_idx, const uint16_t* x,
                         int32_t* counts, int32_t* offsets, int32_t* dest, int32_t* row_token,
                         int32_t* row_slot, uint16_t* Xp, void* stream);

/* Multi-rank form of the token mapping (UniEP page, section 2.2,
 * Algorithm 1): this rank's slots get addresses
 *   dest[t*k+j] = rank_base[e] + (stable rank of slot t*k+j among this
 *                 rank's slots routed to e),   e = topk_idx[t*k+j],
 * where rank_base[e] (device, [E]) is the start of expert e's segment in its
 * owner's receive buffer plus the slots that lower ranks send to e -- the
 * prefix sums over the all-gathered per-rank counts.  counts [E] and
 * offsets [E+1] receive this rank's own counts and their exclusive scan
 * (the values to all-gather).  rank_base = NULL gives the single-rank
 * mapping (dest equals moe_dispatch's).  Uses the histogram scratch of ws
 * only. */
int moe_token_addresses(const moe_cfg* cfg, const int32_t* topk_idx, const int32_t* rank_base,
                        int32_t* counts, int32_t* offsets, int32_t* dest, void* ws, void* stream);

/* Cross-rank bases of the multi-rank token mapping (UniEP page, section 2.2,
 * Algorithm 1: the per-expert counts of every rank are all-gathered, and
 * each rank's slots to expert e are placed after those of the lower ranks).
 * all_counts [G][E] int32: rank g's slots routed to expert e (each rank's
 * moe_token_addresses counts, gathered in rank order).  owner [E] int32:
 * the rank that holds expert e (values outside [0, G) are clamped); the
 * experts of one owner are laid out in its receive buffer in index order.
 * Writes rank_base [E] for rank `rank`:
 *   rank_base[e] = sum of all ranks' counts of the experts u < e with
 *                  owner[u] == owner[e]  +  sum over g < rank of counts[g][e]
 * (the input moe_token_addresses takes), and, if recv_rows [G] is non-NULL,
 * the rows each owner receives.  Device memory, one small launch on
 * `stream`; every sum runs in ascending order, so the result is exact
 * (int32: the total rows per owner must stay below 2^31).
 * Limits: 1 <= E <= 256, 1 <= G <= 65536, 0 <= rank < G (MOE_ERR_SHAPE). */
int moe_rank_bases(const int32_t* all_counts, int G, int E, const int32_t* owner, int rank,
                   int32_t* rank_base, int32_t* recv_rows, void* stream);

/* Expert FFN as two grouped GEMMs over the ragged expert segments
 * (UniEP page, section 1.1 "GroupGEMM -> SwiGLU -> GroupGEMM"; padding-free
 * grouped GEMM with per-segment pointer arithmetic, section 2.2).
 * GEMM 1, per GEMM row r of segment e (A row = Xp[r], or x[t] for shared
 * rows):  a = A.W1_e^T, b = A.W3_e^T accumulated in fp32;
 *         Hw[r] = bf16(w_r * (silu(a) * b)), silu(a) = a / (1 + exp(-a)),
 *         rounded once from fp32, with w_r = topk_w[row_slot[r]] for routed
 *         rows and 1 for shared rows (the gate score applied before the
 *         down projection, which is linear).
 *         If AB is non-NULL, AB[r] = [bf16(a) | bf16(b)]  ([R_s, 2f]).
 * GEMM 2: O'[r] = fl32(Hw[r].W2_e^T).  Hw [R_s, f] bf16, O' [R_s, d] fp32.
 *         Experts with no rows are skipped.
 * offsets/row_slot come from moe_dispatch. */
int moe_group_gemm_swiglu(const moe_cfg* cfg, const uint16_t* Xp, const uint16_t* x,
                          const int32_t* offsets, const int32_t* row_slot,
                          const float* topk_w, const uint16_t* W1, const uint16_t* W3,
                          const uint16_t* W2, uint16_t* Hw, uint16_t* AB, float* Oprime,
                          void* ws, void* stream);

/* Combine (UniEP page, section 1.1: weighted sum by gate score; the
 * weight is already applied in O').  y [T, d] fp32:
 *   y[t] = ((O'[dest[t*k]] + O'[dest[t*k+1]]) + ... + O'[dest[t*k+k-1]])
 *          + O'[R + t] + ... + O'[R + (S-1)*T + t]
 * summed in exactly this order in fp32, so y is bitwise reproducible. */
int moe_combine(const moe_cfg* cfg, const float* Oprime, const int32_t* dest,
                float* y, void* ws, void* stream);

/* Whole forward: route -> dispatch -> GEMM 1 -> GEMM 2 -> combine.
 * Outputs y [T, d] fp32, topk_idx [T, k], topk_w [T, k]; the routing tables
 * and activations are kept in `ws` for moe_layer_bwd.  use_megakernel = 1
 * runs dispatch..combine as one persistent launch that claims tasks from an
 * atomic ticket counter and orders them with device-side readiness counters
 * (UniEP page, section 2.2: persistent workers, scoreboard, dynamic SM
 * scheduling); its outputs are bitwise equal to use_megakernel = 0.  Its
 * tiles run on CTA pairs like the stand-alone GEMMs (see
 * moe_set_gemm_pair_kinds): the pair's even CTA claims each ticket and
 * hands it to the odd one, and the pair splits each gather task.
 * use_megakernel = 1 needs d_model <= 24576 (a gathered row fits a pipeline
 * stage; MOE_ERR_SHAPE otherwise).
 * Route and the permutation tables run as one cooperative launch with grid
 * barriers between histogram, scan and scatter (see moe_set_route_fusion). */
int moe_layer_fwd(const moe_cfg* cfg, const float* logits, const uint16_t* x,
                  const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                  float* y, int32_t* topk_idx, float* topk_w, void* ws,
                  int use_megakernel, void* stream);

/* ---------------------------------------------------------------- backward
 * Gradients of a loss L given dy = dL/dy (bf16 [T, d]).  The backward is the
 * mirror of the forward plus the transposed GroupGEMM for the weight
 * gradients (UniEP page, section 1.1); it splits into the input-gradient
 * part (B) and the weight-gradient part (W) (GraphPP page, sections 2 and
 * 5.1). */

/* Combine backward: G[r] = dy[row_token[r]] for the R routed rows (bf16,
 * exact copy; shared rows read dy directly). */
int moe_combine_bwd(const moe_cfg* cfg, const uint16_t* dy, const int32_t* row_token,
                    uint16_t* G, void* ws, void* stream);

/* Expert FFN backward.  For GEMM row r (token t, weight w_r, expert e):
 *   dHraw = dy_t . W2_e            (fp32 accumulate, K = d)
 *   a, b = the bf16 values in AB[r];  s = sigmoid(a)
 *   dH = w_r * dHraw
 *   dA = dH * b * s * (1 + a * (1 - s));  dB = dH * a * s
 *   dAB[r] = [bf16(dA) | bf16(dB)]          ([R_s, 2f])
 *   dw[t, j] = <dHraw, a * s * b> for routed rows (= <dy_t, unscaled o_r>
 *              with h formed again from the saved a and b),
 *              summed over fixed column tiles in tile order      ([T, k])
 *   dXp[r] = dA . W1_e + dB . W3_e          (fp32 [R_s, d], K = 2f)
 *   dW1_e = sum_r dA_r^T A_r, dW3_e = sum_r dB_r^T A_r   (fp32 [E+S, f, d])
 *   dW2_e = sum_r dy_t^T Hw_r                              (fp32 [E+S, d, f])
 * where A_r = Xp[r] (routed) or x[t] (shared); each weight-gradient sum
 * runs over the segment's rows in ascending order inside one CTA (no
 * split-K atomics), and experts with no rows get exact zeros.
 * which: 1 = input part (dAB, dw, dXp), 2 = weight part (dW1, dW3, dW2;
 * needs dAB from a previous which=1 call), 3 = both.
 * G from moe_combine_bwd; AB, Hw from moe_group_gemm_swiglu. */
int moe_group_gemm_swiglu_bwd(const moe_cfg* cfg, const uint16_t* G, const uint16_t* dy,
                              const uint16_t* Xp, const uint16_t* x,
                              const int32_t* offsets, const int32_t* row_slot,
                              const int32_t* dest, const float* topk_w,
                              const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                              const uint16_t* Hw, const uint16_t* AB,
                              uint16_t* dAB, float* dw, float* dXp,
                              float* dW1, float* dW3, float* dW2, int which,
                              void* ws, void* stream);

/* Dispatch backward: dx[t] = sum over j in slot order of dXp[dest[t*k+j]],
 * then + dXp[R + s*T + t] for s = 0..S-1, fp32 (same order as combine). */
int moe_dispatch_bwd(const moe_cfg* cfg, const float* dXp, const int32_t* dest,
                     float* dx, void* ws, void* stream);

/* Router backward.  dw [T, k] = dL/dw.  p recomputed from the logits
 * exactly as moe_route computes it.
 *   renorm = 0: dlogits_i = p_i * (dw_{j(i)} [i picked] - sum_j dw_j w_j)
 *   renorm = 1: dlogits_i = w_{j(i)} (dw_{j(i)} - sum_j dw_j w_j) if i
 *               was picked, else 0.
 * The top-k choice itself is piecewise constant and has no gradient. */
int moe_route_bwd(const moe_cfg* cfg, const float* logits, const int32_t* topk_idx,
                  const float* topk_w, const float* dw, float* dlogits,
                  void* ws, void* stream);

/* Whole backward from the state moe_layer_fwd left in `ws`.
 * which: 1 = dx and dlogits only (B part), 2 = dW1, dW3, dW2 only (W part;
 * needs a previous which=1 or 3 call on the same ws), 3 = everything.
 * Plus MOE_BWD_MEGAKERNEL: the B part's combine-bwd gather, dH GEMM, dX GEMM
 * and slot-order dx sum run as one persistent MegaKernel launch (UniEP page,
 * section 2.2: its MegaKernels serve the backward steps too), with the same
 * ticket cursor and readiness counters as the forward one; the dw reduce and
 * router backward follow as two small launches.  Same bits as without.
 * Outputs not requested may be NULL. */
#define MOE_BWD_MEGAKERNEL 4
int moe_layer_bwd(const moe_cfg* cfg, const uint16_t* dy, const float* logits,
                  const uint16_t* x, const uint16_t* W1, const uint16_t* W3,
                  const uint16_t* W2, const int32_t* topk_idx, const float* topk_w,
                  void* ws, float* dx, float* dlogits, float* dW1, float* dW3,
                  float* dW2, int which, void* stream);

/* Reads the device error word of `ws` into *code (MOE_OK or a negative
 * MOE_ERR_*) and *info (a code-specific detail, e.g. the token of a
 * non-finite logit or the task of a timed-out wait).  Synchronises
 * `stream` only. */
int moe_get_device_error(const void* ws, void* stream, int* code, int* info);

/* Number of SMs of the current device as the library sees it (grid size of
 * its persistent kernels). */
int moe_num_sms(void);

/* Caps the number of CTAs of the persistent kernels (grouped GEMMs, the
 * MegaKernel and the fused routing launch) at n; n <= 0 restores one CTA per SM.  Results never depend
 * on it (each output element has one fixed producer and reduction order);
 * it exists to test exactly that.  Process-wide, not thread-safe. */
int moe_set_grid_limit(int n);

/* Fused routing of moe_layer_fwd.  On (the default), the router, the
 * per-block expert histogram, the scan and the stable scatter run as one
 * cooperative launch (every CTA resident; two grid barriers, each a bounded
 * wait that sets MOE_ERR_TIMEOUT rather than hang; the barrier state lives in
 * the error region, so after a timeout call moe_ws_init).  Off, or where the
 * device refuses the cooperative launch, they run as three kernels.  The
 * tables are bitwise the same either way, and the CTA cap of
 * moe_set_grid_limit applies to this launch too.  Returns the previous
 * setting.  Process-wide, not thread-safe. */
int moe_set_route_fusion(int on);

/* B/W overlap of moe_layer_bwd with which == 3 (GraphPP page, section 2:
 * input gradients B on the critical path, weight gradients W deferrable).
 * On (the default), the dW GEMMs run on a second stream that the library
 * owns (one per device, created on first use, kept until exit), forked from
 * the caller's stream after the dH GEMM and joined back before the call
 * returns, so the caller's stream still orders everything; they then fill
 * the SMs that the dX GEMM's tail frees and that the memory-bound dx sum and
 * router backward leave idle.  Off runs everything on the caller's stream.
 * The bits are the same either way.  Returns the previous setting.
 * Process-wide, not thread-safe. */
int moe_set_bwd_overlap(int on);

/* Backward GEMMs of moe_layer_bwd with which == 3 (without
 * MOE_BWD_MEGAKERNEL).  On, dX, dW1/dW3 and dW2 run as one persistent
 * launch whose single ticket counter interleaves their tiles: dX's tiles are
 * spread evenly over the tickets, and the weight-gradient tiles fill the rest,
 * longest segments first.  The tensor-heavy dX tiles and the write-heavy
 * short-K weight-gradient tiles then share the SMs and the memory system
 * instead of taking turns (GraphPP page, section 2: the W part is deferrable
 * work that can fill the B part's gaps; UniEP page, section 2.2: dynamic SM
 * scheduling over one task space).  The dw reduce and router backward run
 * before it, and the dx sum after it, on the caller's stream.  Off (the
 * default): dX, then the weight-gradient GEMMs on the B/W overlap's second
 * stream.  Same bits either way.  The one launch is shorter than the
 * three kernels back to back, but the whole step measured slower than the
 * default at every layer tried, since the default overlaps the W GEMMs with
 * dX and the dx sum.  Returns the previous setting.
 * Process-wide, not thread-safe. */
int moe_set_bwd_fused_gemms(int on);

/* Selects, per grouped-GEMM kind, the tile shape: bit k of `mask` set runs
 * kind k on CTA pairs (thread-block clusters of two; the pair computes a
 * 256 x 256 tile with tcgen05 MMAs of the CTA group of two, each CTA holding
 * half of A and half of B); clear runs it one CTA per 128 x 256 tile.  Bits:
 * 0 GEMM 1 (gate/up), 1 GEMM 2 (down), 2 dH, 3 dX, 4 dW1/dW3, 5 dW2.  The
 * default is all six, what measures fastest on a DeepSeek-V2-Lite-like
 * layer (T=8192, d=2048, f=1408, E=64, k=6, S=2); moe_autotune picks per
 * layer.  The MegaKernels follow it: the forward one runs on CTA pairs when
 * bits 0 and 1 are set, the backward one when bits 2 and 3 are (and a row
 * of d_model bf16 fits a 32 KB pipeline stage), else one CTA per tile.
 * Results are the same bits either way: every output element is the same
 * fp32 sum over K in the same order.  Returns the previous mask.
 * Process-wide, not thread-safe. */
int moe_set_gemm_pair_kinds(int mask);

/* Prefetch depth of grouped-GEMM kind `kind` (numbered as above): while a
 * CTA loads a tile, it brings the first `kblocks` K blocks (64 deep) of its
 * next tile into L2 (0 = none; clamped to [0, 64]).  A performance knob only:
 * results are unchanged.  Returns the previous depth, or MOE_ERR_ARG for an
 * unknown kind.  Process-wide, not thread-safe. */
int moe_set_gemm_prefetch(int kind, int kblocks);

/* Tile order of the weight-gradient grouped GEMMs (kinds 4 dW1/dW3 and 5
 * dW2, numbered as above).  order 0 (the default): tiles handed out longest
 * segments first.  order 1: the tiles of the long segments (more than twice
 * the mean rows of the non-empty segments, e.g. the shared experts) are
 * spread evenly over the first three quarters of the tickets, between the
 * short segments' tiles, so compute-heavy tiles (long K, few output bytes per
 * flop) and write-heavy ones (short K, the same fp32 output per tile) run
 * side by side.  A performance knob only: each output element keeps its one
 * producer and its K order.  Returns the previous order, or MOE_ERR_ARG for
 * another kind or order.  Process-wide, not thread-safe. */
int moe_set_gemm_tile_order(int kind, int order);

/* Epilogue stores of the fp32-output grouped GEMMs (kinds 1 GEMM 2, 3 dX,
 * 4 dW1/dW3, 5 dW2).  direct 0 (the default): each warp stages its rows
 * through shared memory and a TMA tensor store writes them.  direct 1: the
 * accumulator is read in a 16-lane shape and written straight from
 * registers, 64 contiguous bytes per row and store, sparing the shared
 * memory traffic of the staging; the staging memory then holds one more
 * pipeline stage on CTA pairs (see moe_gemm_max_stages).  Same values
 * either way.  Returns the
 * previous mode, or MOE_ERR_ARG for another kind or mode.  Process-wide,
 * not thread-safe. */
int moe_set_gemm_epilogue(int kind, int direct);

/* Pipeline stages (shared-memory ring slots of one 64-deep K block each) of
 * grouped-GEMM kind `kind`: 0 = as many as fit (the default), else at least
 * 2 and at most moe_gemm_max_stages().  A performance knob only.  Returns
 * the previous request, or MOE_ERR_ARG.  Process-wide, not thread-safe. */
int moe_set_gemm_stages(int kind, int stages);
/* Stages that fit for `kind` with cta_group (1 or 2) CTAs per tile and the
 * kind's current epilogue stores (moe_set_gemm_epilogue: 6 on pairs, 7 for
 * an fp32-output kind with direct stores; 4 on single CTAs); 0 for an
 * unknown kind or group. */
int moe_gemm_max_stages(int kind, int cta_group);

/* ------------------------------------------------------------ autotuner
 * UniEP page ("Unified Expert-Parallel MoE MegaKernel for LLM Training"),
 * section 3 names autotuning and an analytical model without giving their
 * content.  moe_autotune measures instead, on the caller's own layer
 * (forward + backward), coordinate-wise:
 *  1. per grouped-GEMM kind, the tile shape (one CTA per tile or CTA pairs)
 *     x the next-tile L2 prefetch depth (0, 4 or 8 K blocks);
 *  2. the weight-gradient kinds' tile order (longest first or interleaved),
 *     then the fp32-output kinds' epilogue stores (staged or direct);
 *  3. the pipeline depth (as many stages as fit, or one fewer);
 *  4. kernel chain against MegaKernel, forward and backward.
 * Phases 1-3 are applied process-wide (moe_set_gemm_pair_kinds,
 * moe_set_gemm_prefetch, moe_set_gemm_tile_order, moe_set_gemm_epilogue,
 * moe_set_gemm_stages);
 * phase 4 is reported for the caller's use_megakernel / MOE_BWD_MEGAKERNEL
 * arguments.  The library's defaults are timed first, and a later candidate
 * replaces the one kept only if it is more than 1% faster, so near ties
 * (within run-to-run spread) do not flip the choice.
 *
 * Arguments are those of moe_layer_fwd and moe_layer_bwd (all device memory
 * owned by the caller, layouts as there); every output and `ws` are
 * overwritten as by a normal forward + backward.  `reps` timed steps per
 * candidate (0 = 2), after one warm-up step each, with the backward's B/W
 * overlap off (restored afterwards) so each kernel is timed alone.
 * Synchronizes `stream` (host-blocking) and resets the kernel-timing totals
 * (moe_trace_*).
 * Choices never change results: the outputs after tuning are the same bits.
 * On error the previous settings are restored and the error is returned. */
typedef struct {
  int pair[6];         /* per kind (numbered as above): 1 = CTA pairs */
  int prefetch_kb[6];  /* per kind: next-tile K blocks prefetched into L2 */
  float us[6];         /* per kind: measured microseconds per launch of the choice */
  int tile_order[6];   /* per kind: tile order (kinds 4, 5; 0 for the others) */
  int stages[6];       /* per kind: pipeline stages in use */
  int epi_direct[6];   /* per kind: 1 = direct epilogue stores (kinds 1, 3, 4, 5) */
  int fwd_megakernel;  /* 1: the forward MegaKernel measured faster than the kernel chain */
  int bwd_megakernel;  /* 1: the backward input-part MegaKernel measured faster */
  float fwd_us[2];     /* forward per call: kernel chain, MegaKernel (microseconds) */
  float bwd_us[2];     /* backward per call: kernel chain, MegaKernel */
} moe_tune_result;

int moe_autotune(const moe_cfg* cfg, const float* logits, const uint16_t* x,
                 const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                 const uint16_t* dy, float* y, int32_t* topk_idx, float* topk_w,
                 float* dx, float* dlogits, float* dW1, float* dW3, float* dW2,
                 void* ws, int reps, void* stream, moe_tune_result* out);

/* Number of CTA pairs of grouped-GEMM kind `kind` (numbered as above) that
 * the current device holds at once; the pair-mode launches use that many
 * pairs (fewer under moe_set_grid_limit).  Returns 0 for an unknown kind or
 * when the query fails. */
int moe_gemm_pair_capacity(int kind);

/* ------------------------------------------------------- kernel timing
 * Optional profiling aid.  While enabled, every kernel launch the library
 * makes is bracketed by a pair of CUDA events recorded on the launching
 * stream (no device memory is allocated; events come from a host pool).
 * moe_trace_read() waits for the recorded events of that kind and returns
 * the summed device time in milliseconds and the number of launches since
 * the last moe_trace_reset().  Process-wide; thread-safe. */
enum {
  MOE_K_ROUTE = 0,        /* router (+ per-block expert histogram) */
  MOE_K_HIST = 1,         /* histogram of caller-given expert indices */
  MOE_K_SCAN = 2,         /* flat exclusive scan -> offsets, bases */
  MOE_K_SCATTER = 3,      /* stable in-block ranks -> dest, row_token, row_slot */
  MOE_K_GATHER = 4,       /* dispatch gather Xp[r] = x[row_token[r]] */
  MOE_K_GEMM1 = 5,        /* grouped GEMM gate/up + SiLU*mul */
  MOE_K_GEMM2 = 6,        /* grouped GEMM down + routing-weight scale */
  MOE_K_COMBINE = 7,      /* slot-order fp32 combine */
  MOE_K_COMBINE_BWD = 8,  /* G[r] = dy[row_token[r]] */
  MOE_K_GEMM_DH = 9,      /* grouped GEMM dy.W2 + SwiGLU backward */
  MOE_K_DW_REDUCE = 10,   /* dw from per-tile partial dots */
  MOE_K_ROUTE_BWD = 11,   /* router backward */
  MOE_K_GEMM_DX = 12,     /* grouped GEMM [dA|dB].[W1;W3] */
  MOE_K_DISPATCH_BWD = 13,/* slot-order fp32 dx sum */
  MOE_K_GEMM_DW13 = 14,   /* ragged-K grouped GEMM dW1, dW3 */
  MOE_K_GEMM_DW2 = 15,    /* ragged-K grouped GEMM dW2 */
  MOE_K_MEGAKERNEL = 16,  /* forward MegaKernel */
  MOE_K_MEGAKERNEL_BWD = 17, /* backward (input-gradient) MegaKernel */
  MOE_K_ROUTE_TABLES = 18, /* router + histogram + scan + scatter, one launch */
  MOE_K_BWD_GEMMS = 19,   /* dX, dW1/dW3 and dW2 interleaved in one launch */
  MOE_K_COUNT = 20
};
/* Testing aid for failure detection (no device fault involved): the forward
 * MegaKernel claims task `ticket` but never runs or signals it, so the
 * tasks that depend on it run into their bounded waits; the kernel then
 * records MOE_ERR_TIMEOUT in the device error word and returns, and the
 * CUDA context stays usable.  ticket < 0 disables it (the default).
 * Process-wide, not thread-safe; never set in normal use. */
int moe_debug_skip_megakernel_task(int ticket);

/* Profiling aid: per-task timeline of the forward MegaKernel.  While `buf`
 * (device memory, 16-byte aligned, at least grid * records_per_cta * 24
 * bytes; grid = moe_num_sms() unless capped) is set, every MegaKernel launch
 * writes, per CTA, up to records_per_cta/2 records for its producer and as
 * many for its first epilogue warp: three u64 each,
 *   [ticket | role << 32 | cta << 40, start ns, end ns]  (%globaltimer),
 * role 0 = producer (claim .. loads issued / gather done), role 1 =
 * epilogue (task popped .. results published).  Unused records keep their
 * previous contents.  buf = NULL turns it off.  Process-wide. */
int moe_debug_megakernel_trace(void* buf, int records_per_cta);

int moe_trace_enable(int on);
int moe_trace_reset(void);
int moe_trace_read(int kind, double* total_ms, int* launches);
const char* moe_trace_kind_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */

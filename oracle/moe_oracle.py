"""CPU fp64 oracle for one Mixture-of-Experts layer.  TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import or run this module.  The CUDA library never
calls it and shares no code with it.

It is the plain definition of the layer that UniEP fuses into a MegaKernel
(UniEP page, "Unified Expert-Parallel MoE MegaKernel for LLM Training",
section 1.1 and Figure 1): a gating network gives every token a probability
per expert, top-k picks the target experts, the tokens are reordered
(scattered) to their experts, each expert runs GroupGEMM -> SwiGLU ->
GroupGEMM back to the model width, and the results return and are summed
weighted by the gate score.  The backward pass mirrors the forward and needs
the transposed GroupGEMM for the weight gradients (same section).  The SwiGLU
expert is the MLP of the GraphPP page, section 5.1-5.2 (gate projection w1,
up projection w3, SiLU, gate product, down projection w2; grad_w2 from the
hidden activation and grad_out, grad_w1/w3 from x and the intermediate
gradients, grad_x as the sum of the two paths).

Every value is computed in float64 from the exact bf16/fp32 input bits.  No
intermediate is rounded.  Matrix products use numpy's matmul as a library
step; there is no blocking or reordering beyond the definitions below.

Readings taken where the pages are silent:
  * softmax over all E experts, then top-k; the routing weight is the
    probability itself (renorm=0) or renormalised over the k picks (renorm=1);
  * top-k is chosen on the fp32 logits, larger first, ties to the lower expert
    index, and -0.0 equals +0.0; slot j holds the j-th pick;
  * the token order inside an expert's segment is the stable order of the
    flat slot index t*k + j (Algorithm 1 with a single rank: base offset 0);
  * shared experts are always-on SwiGLU experts with weight 1, stored after
    the routed experts, added after the routed slots in shared-index order;
  * no biases, no capacity limit: every slot is computed.

Parity pins: every public function here is pinned by ``tests/test_oracle.py``
(hand-enumerated routing case, library sort, closed forms, dense SwiGLU via
torch float64, torch float64 autograd and central finite differences).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
from scipy.special import expit


class NonFiniteLogits(ValueError):
    """Raised when a router logit is NaN or infinite."""


def f64(a) -> np.ndarray:
    """Exact widening of a numpy array or a CPU torch tensor (any float
    dtype, bf16 included) to float64."""
    if hasattr(a, "detach"):  # torch tensor
        import torch
        return a.detach().to(torch.float64).cpu().numpy()
    return np.asarray(a, dtype=np.float64)


def take_rows(a, idx) -> np.ndarray:
    """Rows ``idx`` of a numpy array or CPU torch tensor, widened to float64."""
    if hasattr(a, "detach"):
        import torch
        return f64(a[torch.as_tensor(np.asarray(idx, dtype=np.int64))])
    return f64(np.asarray(a)[idx])


# --------------------------------------------------------------------------
# Gating: softmax over experts, then top-k (UniEP page, section 1.1).
# --------------------------------------------------------------------------
def softmax(z: np.ndarray) -> np.ndarray:
    """Row softmax p_i = exp(z_i - m) / sum_j exp(z_j - m), m = max_j z_j."""
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=1, keepdims=True)


def topk_select(z: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per row, larger first, ties to the
    lower index.  A stable sort of -z keeps equal values (-0.0 == +0.0) in
    index order."""
    return np.argsort(-z, axis=1, kind="stable")[:, :k].astype(np.int64)


@dataclass
class Routing:
    p: np.ndarray    # [T, E] softmax probabilities
    sel: np.ndarray  # [T, k] selected experts, slot order
    w: np.ndarray    # [T, k] routing weights


def route(logits, k: int, renorm: int = 0) -> Routing:
    """Gate: probabilities over all experts, top-k experts, routing weights."""
    z = f64(logits)
    if not np.all(np.isfinite(z)):
        raise NonFiniteLogits("router logits contain NaN or Inf")
    p = softmax(z)
    sel = topk_select(z, k)
    w = np.take_along_axis(p, sel, axis=1)
    if renorm:
        w = w / w.sum(axis=1, keepdims=True)
    return Routing(p, sel, w)


# --------------------------------------------------------------------------
# Deterministic token mapping (UniEP page, section 2.2, Algorithm 1, with a
# single rank so the cross-rank base offset is zero).
# --------------------------------------------------------------------------
@dataclass
class Permutation:
    counts: np.ndarray     # [E]    slots routed to each expert
    offsets: np.ndarray    # [E+1]  exclusive prefix sum of counts
    dest: np.ndarray       # [T*k]  flat slot t*k+j -> permuted row
    row_token: np.ndarray  # [T*k]  permuted row -> token
    row_slot: np.ndarray   # [T*k]  permuted row -> flat slot t*k+j


def permute(sel: np.ndarray, E: int) -> Permutation:
    """Stable grouping of the flat slots by expert: expert e's segment holds
    its slots in ascending flat-slot order (ascending token, then slot)."""
    T, k = sel.shape
    flat = np.asarray(sel).reshape(-1)
    per_expert = [np.nonzero(flat == e)[0] for e in range(E)]
    counts = np.array([len(s) for s in per_expert], dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    row_slot = (np.concatenate(per_expert) if T * k else np.zeros(0)).astype(np.int64)
    row_token = row_slot // k
    dest = np.empty(T * k, dtype=np.int64)
    dest[row_slot] = np.arange(T * k, dtype=np.int64)
    return Permutation(counts, offsets, dest, row_token, row_slot)


# --------------------------------------------------------------------------
# SwiGLU expert (GraphPP page, section 5.1-5.2 MLP; UniEP page, section 1.1).
# --------------------------------------------------------------------------
def silu(a: np.ndarray) -> np.ndarray:
    """silu(a) = a * sigmoid(a)."""
    return a * expit(a)


def swiglu_expert(xr: np.ndarray, W1e: np.ndarray, W3e: np.ndarray, W2e: np.ndarray):
    """Rows xr [n, d] through one expert; W1e, W3e [f, d], W2e [d, f]
    (nn.Linear [out, in] layout).  Returns a, b, h, o."""
    a = xr @ W1e.T
    b = xr @ W3e.T
    h = silu(a) * b
    o = h @ W2e.T
    return a, b, h, o


@dataclass
class Segment:
    """Rows of one expert in the GEMM row space [0, R + S*T)."""
    expert: int        # weight index (shared experts follow the routed ones)
    rows: np.ndarray   # row ids in the GEMM row space
    tokens: np.ndarray # token of every row
    weight: np.ndarray # routing weight of every row (1 for shared rows)


def segments(routing: Routing, perm: Permutation, E: int, S: int, T: int):
    """Routed segments in expert order, then one segment per shared expert
    (rows R + s*T + t, token order)."""
    k = routing.sel.shape[1]
    R = T * k
    w_flat = routing.w.reshape(-1)
    out = []
    for e in range(E):
        rows = np.arange(perm.offsets[e], perm.offsets[e + 1])
        out.append(Segment(e, rows, perm.row_token[rows], w_flat[perm.row_slot[rows]]))
    for s in range(S):
        out.append(Segment(E + s, R + s * T + np.arange(T), np.arange(T), np.ones(T)))
    return out


@dataclass
class Forward:
    routing: Routing
    perm: Permutation
    segs: list
    a: np.ndarray   # [R_s, f]
    b: np.ndarray   # [R_s, f]
    h: np.ndarray   # [R_s, f]
    o: np.ndarray   # [R_s, d] unscaled expert outputs
    y: np.ndarray   # [T, d]


def layer_fwd(x, logits, W1, W3, W2, k: int, S: int = 0, renorm: int = 0,
              expert_fn=None) -> Forward:
    """y_t = sum_j w_tj * Expert_{sel_tj}(x_t) + sum_s Shared_s(x_t).

    ``expert_fn(xr, e) -> o`` replaces the SwiGLU expert (used to pin the
    dispatch/combine machinery with identity experts)."""
    x = f64(x)
    W1, W3, W2 = f64(W1), f64(W3), f64(W2)
    T, d = x.shape
    E = np.asarray(logits).shape[1]
    f = W1.shape[1]
    routing = route(logits, k, renorm)
    perm = permute(routing.sel, E)
    segs = segments(routing, perm, E, S, T)
    Rs = T * k + S * T
    a = np.zeros((Rs, f)); b = np.zeros((Rs, f)); h = np.zeros((Rs, f))
    o = np.zeros((Rs, d))
    for sg in segs:
        xr = x[sg.tokens]
        if expert_fn is not None:
            o[sg.rows] = expert_fn(xr, sg.expert)
            continue
        a[sg.rows], b[sg.rows], h[sg.rows], o[sg.rows] = swiglu_expert(
            xr, W1[sg.expert], W3[sg.expert], W2[sg.expert])
    # Combine: weighted sum over the k slots of each token, then shared rows.
    y = np.zeros((T, d))
    dest = perm.dest.reshape(T, k)
    for j in range(k):
        y += routing.w[:, j:j + 1] * o[dest[:, j]]
    for s in range(S):
        y += o[T * k + s * T + np.arange(T)]
    return Forward(routing, perm, segs, a, b, h, o, y)


# --------------------------------------------------------------------------
# Backward (UniEP page, section 1.1: mirror of the forward plus the
# transposed GroupGEMM for weight gradients; GraphPP page, section 5.1-5.2
# MLP backward).
# --------------------------------------------------------------------------
def dsilu(a: np.ndarray) -> np.ndarray:
    """d silu / da = sigma(a) * (1 + a * (1 - sigma(a)))."""
    s = expit(a)
    return s * (1.0 + a * (1.0 - s))


def route_bwd(routing: Routing, dw: np.ndarray, renorm: int) -> np.ndarray:
    """Gradient of the loss w.r.t. the logits given dL/dw [T, k].

    renorm=0: w_j = p_{e_j}, dp_e/dz_i = p_e (delta_ei - p_i)
              dz_i = p_i * (dw_{j(i)} [i selected] - sum_j dw_j p_{e_j})
    renorm=1: w_j = softmax over the selected logits only
              dz_i = w_{j(i)} (dw_{j(i)} - sum_j dw_j w_j) for i selected, else 0
    The selection itself is piecewise constant and has no gradient."""
    T, E = routing.p.shape
    sel_dw = np.zeros((T, E))
    np.put_along_axis(sel_dw, routing.sel, dw, axis=1)
    if renorm == 0:
        inner = (dw * routing.w).sum(axis=1, keepdims=True)
        return routing.p * (sel_dw - inner)
    inner = (dw * routing.w).sum(axis=1, keepdims=True)
    dz_sel = routing.w * (dw - inner)
    dz = np.zeros((T, E))
    np.put_along_axis(dz, routing.sel, dz_sel, axis=1)
    return dz


@dataclass
class Backward:
    dx: np.ndarray       # [T, d]
    dlogits: np.ndarray  # [T, E]
    dW1: np.ndarray      # [E+S, f, d]
    dW3: np.ndarray      # [E+S, f, d]
    dW2: np.ndarray      # [E+S, d, f]
    dw: np.ndarray       # [T, k]
    # per GEMM row (routed rows in segment order, then shared rows)
    dA: np.ndarray = None    # [R_s, f] dL/da
    dB: np.ndarray = None    # [R_s, f] dL/db
    dXp: np.ndarray = None   # [R_s, d] dL/d(expert input) of the row


def layer_bwd(fw: Forward, dy, x, W1, W3, W2, renorm: int = 0) -> Backward:
    """Gradients of L = <dy, y> for the layer computed by ``layer_fwd``."""
    dy, x = f64(dy), f64(x)
    W1, W3, W2 = f64(W1), f64(W3), f64(W2)
    T, d = x.shape
    k = fw.routing.sel.shape[1]
    nexp, f, _ = W1.shape
    dx = np.zeros((T, d))
    dW1 = np.zeros((nexp, f, d)); dW3 = np.zeros((nexp, f, d)); dW2 = np.zeros((nexp, d, f))
    dw_rows = np.zeros(T * k)
    Rs = fw.a.shape[0]
    dA_rows = np.zeros((Rs, f)); dB_rows = np.zeros((Rs, f)); dXp_rows = np.zeros((Rs, d))
    for sg in fw.segs:
        if len(sg.rows) == 0:
            continue
        g = dy[sg.tokens]                        # dL/dy for every row
        a, b, h, o = fw.a[sg.rows], fw.b[sg.rows], fw.h[sg.rows], fw.o[sg.rows]
        if sg.expert < fw.routing.p.shape[1]:    # routed rows carry a weight
            dw_rows[sg.rows] = (g * o).sum(axis=1)
        wg = sg.weight[:, None] * g              # dL/do
        dh = wg @ W2[sg.expert]                  # dL/dh   [n, f]
        dA = dh * b * dsilu(a)                   # dL/da
        dB = dh * silu(a)                        # dL/db
        dXp = dA @ W1[sg.expert] + dB @ W3[sg.expert]
        dx[sg.tokens] += dXp
        dA_rows[sg.rows], dB_rows[sg.rows], dXp_rows[sg.rows] = dA, dB, dXp
        dW2[sg.expert] = wg.T @ h
        dW1[sg.expert] = dA.T @ x[sg.tokens]
        dW3[sg.expert] = dB.T @ x[sg.tokens]
    dw = dw_rows[fw.perm.dest].reshape(T, k)
    dlogits = route_bwd(fw.routing, dw, renorm)
    return Backward(dx, dlogits, dW1, dW3, dW2, dw, dA_rows, dB_rows, dXp_rows)


# --------------------------------------------------------------------------
# Sampled evaluation for workloads too large to run whole: the same
# definitions restricted to a subset of tokens or of weight-gradient entries.
# --------------------------------------------------------------------------
def tokens_fwd_bwd(x, logits, W1, W3, W2, dy, k: int, S: int, renorm: int, tokens):
    """y, dx and dlogits rows of the given tokens, computed token by token
    group-wise per expert.  Returns (routing of those tokens, y, dx, dlogits,
    dw)."""
    tokens = np.asarray(tokens, dtype=np.int64)
    xs = take_rows(x, tokens)
    dys = take_rows(dy, tokens)
    E = np.asarray(logits).shape[1]
    routing = route(f64(logits)[tokens], k, renorm)
    n, d = xs.shape
    y = np.zeros((n, d)); dx = np.zeros((n, d)); dw = np.zeros((n, k))
    # one pass per expert (only the experts the sampled tokens use, each
    # expert's weights widened once); a token picks an expert at most once
    for e in range(E + S):
        if e < E:
            idx, slot = np.nonzero(routing.sel == e)
            if len(idx) == 0:
                continue
            wgt = routing.w[idx, slot]
        else:
            idx, slot, wgt = np.arange(n), None, np.ones(n)
        W1e, W3e, W2e = f64(W1[e]), f64(W3[e]), f64(W2[e])
        a, b, h, o = swiglu_expert(xs[idx], W1e, W3e, W2e)
        y[idx] += wgt[:, None] * o
        g = dys[idx]
        if slot is not None:
            dw[idx, slot] = (g * o).sum(axis=1)
        dh = (wgt[:, None] * g) @ W2e
        dA = dh * b * dsilu(a); dB = dh * silu(a)
        dx[idx] += dA @ W1e + dB @ W3e
    dlogits = route_bwd(routing, dw, renorm)
    return routing, y, dx, dlogits, dw


def dW_entries(x, logits, W1, W3, W2, dy, k: int, S: int, renorm: int,
               which: str, expert: int, rows, cols, routing: Routing = None, perm: Permutation = None):
    """Selected entries of dW1/dW3 ([expert, n, c]) or dW2 ([expert, c, n]),
    each summed over the expert's whole segment.  ``rows``/``cols`` index the
    weight matrix of that expert.  ``routing``/``perm`` may be passed in when
    already computed for these logits."""
    W1e, W3e, W2e = f64(W1[expert]), f64(W3[expert]), f64(W2[expert])
    T = x.shape[0]
    E = np.asarray(logits).shape[1]
    if expert < E:
        if routing is None:
            routing = route(logits, k, renorm)
        if perm is None:
            perm = permute(routing.sel, E)
        r = np.arange(perm.offsets[expert], perm.offsets[expert + 1])
        tok = perm.row_token[r]
        wgt = routing.w.reshape(-1)[perm.row_slot[r]]
    else:
        tok = np.arange(T); wgt = np.ones(T)
    rows = np.asarray(rows); cols = np.asarray(cols)
    xr = take_rows(x, tok); g = take_rows(dy, tok)
    # The hidden unit n of each entry: the row of dW1/dW3, the column of dW2.
    # The segment-long columns a[:, n], b[:, n] (and dh[:, n]) are formed once
    # per distinct n, all of them in one product with the segment.
    ns, j = np.unique(rows if which in ("W1", "W3") else cols, return_inverse=True)
    a = xr @ W1e[ns].T; b = xr @ W3e[ns].T  # [segment rows, distinct n]
    if which in ("W1", "W3"):
        dh = wgt[:, None] * (g @ W2e[:, ns])
        grad_pre = dh * b * dsilu(a) if which == "W1" else dh * silu(a)
        # dW1/dW3[n, c] = sum over the segment of grad_pre[:, n] * x[:, c]
        return np.einsum("ri,ri->i", grad_pre[:, j], xr[:, cols])
    h = silu(a) * b
    # dW2[m, n] = sum over the segment of (w * g)[:, m] * h[:, n]
    return np.einsum("ri,ri->i", wgt[:, None] * g[:, rows], h[:, j])

"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against something fixed independently of its
code: a routing case enumerated by hand (tests/golden), Python's own sort as
the definition of a stable order, closed forms, a dense SwiGLU MLP written
with torch float64 library calls, a per-token brute force, torch float64
autograd, and central finite differences of the oracle's own forward.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "route_hand_T8E4k2.json")


def _rand_layer(T, d, f, E, k, S=0, seed=0, wstd=0.1):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g, dtype=torch.float64)
    logits = torch.randn(T, E, generator=g, dtype=torch.float64)
    W1 = torch.randn(E + S, f, d, generator=g, dtype=torch.float64) * wstd
    W3 = torch.randn(E + S, f, d, generator=g, dtype=torch.float64) * wstd
    W2 = torch.randn(E + S, d, f, generator=g, dtype=torch.float64) * wstd
    dy = torch.randn(T, d, generator=g, dtype=torch.float64)
    return x, logits, W1, W3, W2, dy


def _py_topk(row, k):
    """Top-k by Python's stable sort on (-value, index)."""
    return sorted(range(len(row)), key=lambda e: (-row[e], e))[:k]


# ---------------------------------------------------------------- routing
@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_case(case):
    z = np.array(case["logits"], dtype=np.float32)
    r = O.route(z, case["k"], renorm=0)
    assert r.sel.tolist() == case["sel"]
    want_w = np.array([[eval(s, {"exp": math.exp}) for s in row] for row in case["w_renorm0_closed_form"]])
    np.testing.assert_allclose(r.w, want_w, rtol=1e-14, atol=0)
    p = O.permute(r.sel, case["E"])
    assert p.counts.tolist() == case["counts"]
    assert p.offsets.tolist() == case["offsets"]
    assert p.row_slot.tolist() == case["row_slot"]
    assert p.row_token.tolist() == case["row_token"]
    assert p.dest.tolist() == case["dest"]


def test_signed_zero_is_a_tie():
    z = np.array([[-0.0, 0.0, -1.0], [0.0, -0.0, -1.0]], dtype=np.float32)
    assert O.route(z, 1).sel[:, 0].tolist() == [0, 0]


@pytest.mark.parametrize("E,k", [(4, 2), (8, 3), (16, 8), (5, 5)])
def test_topk_matches_python_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    # small-integer logits make ties common; sprinkle signed zeros
    z = rng.integers(-3, 4, size=(200, E)).astype(np.float32)
    z[rng.random(z.shape) < 0.1] = -0.0
    r = O.route(z, k)
    for t in range(z.shape[0]):
        assert r.sel[t].tolist() == _py_topk(z[t].tolist(), k)


def test_all_equal_logits_give_uniform_weights():
    for E, k in [(8, 2), (6, 3), (64, 6)]:
        z = np.full((3, E), 0.75, dtype=np.float32)
        r0 = O.route(z, k, renorm=0)
        assert np.all(r0.w == 1.0 / E)
        assert r0.sel[0].tolist() == list(range(k))
        r1 = O.route(z, k, renorm=1)
        np.testing.assert_allclose(r1.w, 1.0 / k, rtol=1e-15)


def test_two_expert_softmax_is_logistic():
    from scipy.special import expit
    rng = np.random.default_rng(3)
    z = rng.normal(size=(50, 2)).astype(np.float32)
    r = O.route(z, 1)
    z64 = z.astype(np.float64)
    top = np.where(z64[:, 0] >= z64[:, 1], 0, 1)
    want = expit(z64[np.arange(50), top] - z64[np.arange(50), 1 - top])
    np.testing.assert_allclose(r.w[:, 0], want, rtol=1e-14)


def test_nonfinite_logits_rejected():
    for bad in (np.nan, np.inf, -np.inf):
        z = np.zeros((2, 4), dtype=np.float32)
        z[1, 2] = bad
        with pytest.raises(O.NonFiniteLogits):
            O.route(z, 2)


# ------------------------------------------------------------ permutation
@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (37, 5, 2), (300, 16, 4), (64, 8, 8)])
def test_permutation_is_library_stable_sort(T, E, k):
    rng = np.random.default_rng(T + E + k)
    sel = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    p = O.permute(sel, E)
    flat = sel.reshape(-1).tolist()
    order = sorted(range(T * k), key=lambda i: (flat[i], i))
    assert p.row_slot.tolist() == order
    # invariants: bijection onto [0, T*k), counts, offsets, token order
    assert sorted(p.dest.tolist()) == list(range(T * k))
    assert np.all(p.dest[p.row_slot] == np.arange(T * k))
    assert p.counts.sum() == T * k and np.all(np.diff(p.offsets) >= 0)
    assert p.offsets[0] == 0 and p.offsets[-1] == T * k
    for e in range(E):
        seg = p.row_token[p.offsets[e]:p.offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)  # one token never picks an expert twice
        assert np.all(sel.reshape(-1)[p.row_slot[p.offsets[e]:p.offsets[e + 1]]] == e)


# ---------------------------------------------------------------- forward
def _torch_mlp(x, W1e, W3e, W2e):
    return F.linear(F.silu(F.linear(x, W1e)) * F.linear(x, W3e), W2e)


def test_dense_swiglu_special_case():
    """E=1, k=1: every token goes to the one expert with weight 1, so the
    layer is a dense SwiGLU MLP."""
    x, logits, W1, W3, W2, _ = _rand_layer(40, 24, 36, 1, 1, seed=1)
    for renorm in (0, 1):
        fw = O.layer_fwd(x, logits, W1, W3, W2, k=1, renorm=renorm)
        want = _torch_mlp(x, W1[0], W3[0], W2[0]).numpy()
        np.testing.assert_allclose(fw.y, want, rtol=1e-12, atol=1e-13)


def test_shared_experts_are_dense_mlps():
    x, logits, W1, W3, W2, _ = _rand_layer(30, 16, 20, 4, 2, S=2, seed=2)
    W2z = W2.clone(); W2z[:4] = 0  # silence the routed experts
    fw = O.layer_fwd(x, logits, W1, W3, W2z, k=2, S=2)
    want = sum(_torch_mlp(x, W1[4 + s], W3[4 + s], W2[4 + s]) for s in range(2)).numpy()
    np.testing.assert_allclose(fw.y, want, rtol=1e-12, atol=1e-13)


def test_identity_experts_return_input():
    """With identity experts and weights that sum to one (renorm=1), dispatch
    followed by combine is the identity."""
    x, logits, W1, W3, W2, _ = _rand_layer(100, 12, 8, 6, 3, seed=3)
    fw = O.layer_fwd(x, logits, W1, W3, W2, k=3, renorm=1, expert_fn=lambda xr, e: xr)
    np.testing.assert_allclose(fw.y, x.numpy(), rtol=0, atol=1e-12)
    # k = E with renorm=0: all probabilities are used and sum to one
    x, logits, W1, W3, W2, _ = _rand_layer(50, 12, 8, 4, 4, seed=4)
    fw = O.layer_fwd(x, logits, W1, W3, W2, k=4, renorm=0, expert_fn=lambda xr, e: xr)
    np.testing.assert_allclose(fw.y, x.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("renorm", [0, 1])
def test_per_token_brute_force(renorm):
    """y_t = sum_j w_tj MLP_{e_tj}(x_t) + sum_s MLP_s(x_t), one token at a
    time, with torch softmax and Python's sort for the routing."""
    T, d, f, E, k, S = 24, 16, 20, 5, 2, 1
    x, logits, W1, W3, W2, _ = _rand_layer(T, d, f, E, k, S=S, seed=5)
    fw = O.layer_fwd(x, logits.float(), W1, W3, W2, k=k, S=S, renorm=renorm)
    p = torch.softmax(logits.float().double(), dim=1)
    for t in range(T):
        picks = _py_topk(logits.float()[t].tolist(), k)
        ws = [p[t, e].item() for e in picks]
        if renorm:
            ws = [w / sum(ws) for w in ws]
        yt = sum(w * _torch_mlp(x[t:t + 1], W1[e], W3[e], W2[e]) for w, e in zip(ws, picks))
        yt = yt + sum(_torch_mlp(x[t:t + 1], W1[E + s], W3[E + s], W2[E + s]) for s in range(S))
        np.testing.assert_allclose(fw.y[t], yt[0].numpy(), rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------- backward
def _autograd_layer(x, logits, W1, W3, W2, dy, k, S, renorm):
    """Forward written with torch ops on leaf tensors; autograd supplies
    every gradient.  The routing decisions come from Python's sort."""
    leaves = [t.clone().requires_grad_(True) for t in (x, logits, W1, W3, W2)]
    xl, zl, W1l, W3l, W2l = leaves
    T, E = logits.shape
    p = torch.softmax(zl, dim=1)
    y = torch.zeros_like(xl)
    rows = []
    for t in range(T):
        picks = _py_topk(logits[t].tolist(), k)
        ws = torch.stack([p[t, e] for e in picks])
        if renorm:
            ws = ws / ws.sum()
        yt = sum(ws[j] * _torch_mlp(xl[t:t + 1], W1l[e], W3l[e], W2l[e]) for j, e in enumerate(picks))
        yt = yt + sum(_torch_mlp(xl[t:t + 1], W1l[E + s], W3l[E + s], W2l[E + s]) for s in range(S))
        rows.append(yt)
    y = torch.cat(rows)
    (y * dy).sum().backward()
    return [l.grad.numpy() for l in leaves]


@pytest.mark.parametrize("renorm,S", [(0, 0), (1, 0), (0, 2), (1, 1)])
def test_backward_matches_autograd(renorm, S):
    T, d, f, E, k = 20, 12, 16, 5, 2
    x, logits, W1, W3, W2, dy = _rand_layer(T, d, f, E, k, S=S, seed=10 + renorm + S)
    fw = O.layer_fwd(x, logits, W1, W3, W2, k=k, S=S, renorm=renorm)
    bw = O.layer_bwd(fw, dy, x, W1, W3, W2, renorm=renorm)
    gx, gz, g1, g3, g2 = _autograd_layer(x, logits, W1, W3, W2, dy, k, S, renorm)
    for got, want in [(bw.dx, gx), (bw.dlogits, gz), (bw.dW1, g1), (bw.dW3, g3), (bw.dW2, g2)]:
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_backward_matches_finite_differences():
    """Central differences of L = <dy, y> through the oracle's own forward."""
    T, d, f, E, k, S = 16, 8, 12, 4, 2, 1
    x, logits, W1, W3, W2, dy = _rand_layer(T, d, f, E, k, S=S, seed=20, wstd=0.3)
    args = dict(x=x.numpy(), logits=logits.numpy(), W1=W1.numpy(), W3=W3.numpy(), W2=W2.numpy())
    fw = O.layer_fwd(k=k, S=S, renorm=0, **args)
    bw = O.layer_bwd(fw, dy, x, W1, W3, W2, renorm=0)
    grads = {"x": bw.dx, "logits": bw.dlogits, "W1": bw.dW1, "W3": bw.dW3, "W2": bw.dW2}
    rng = np.random.default_rng(0)
    h = 1e-6
    dyn = dy.numpy()
    for name in grads:
        for _ in range(6):
            idx = tuple(rng.integers(0, s) for s in args[name].shape)
            plus = {kk: v.copy() for kk, v in args.items()}
            minus = {kk: v.copy() for kk, v in args.items()}
            plus[name][idx] += h
            minus[name][idx] -= h
            lp = (O.layer_fwd(k=k, S=S, renorm=0, **plus).y * dyn).sum()
            lm = (O.layer_fwd(k=k, S=S, renorm=0, **minus).y * dyn).sum()
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grads[name][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grads[name][idx])


# ------------------------------------------------------ sampled evaluators
def test_sampled_evaluators_agree_with_full_layer():
    T, d, f, E, k, S = 60, 16, 24, 6, 2, 1
    x, logits, W1, W3, W2, dy = _rand_layer(T, d, f, E, k, S=S, seed=30)
    z = logits.float()
    fw = O.layer_fwd(x, z, W1, W3, W2, k=k, S=S)
    bw = O.layer_bwd(fw, dy, x, W1, W3, W2)
    toks = np.array([0, 7, 13, 59, 31])
    _, y, dx, dz, dw = O.tokens_fwd_bwd(x, z.numpy(), W1, W3, W2, dy, k, S, 0, toks)
    np.testing.assert_allclose(y, fw.y[toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dx, bw.dx[toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dz, bw.dlogits[toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dw, bw.dw[toks], rtol=1e-12, atol=1e-13)
    rng = np.random.default_rng(1)
    for which, full in [("W1", bw.dW1), ("W3", bw.dW3), ("W2", bw.dW2)]:
        for e in range(E + S):
            # repeated rows and columns: entries that share a hidden unit
            rows = np.concatenate([rng.integers(0, full.shape[1], 5), [1, 1, 1]])
            cols = np.concatenate([rng.integers(0, full.shape[2], 5), [2, 0, 2]])
            got = O.dW_entries(x, z.numpy(), W1, W3, W2, dy, k, S, 0, which, e, rows, cols)
            np.testing.assert_allclose(got, full[e][rows, cols], rtol=1e-12, atol=1e-13)

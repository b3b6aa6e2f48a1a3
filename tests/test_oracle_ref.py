"""The numpy oracle against a second, independent implementation of the same
layer: plain C++ loops in fp64 (oracle/moe_oracle_ref.cpp), sharing no code
with it.  Both take the same bf16 / fp32 inputs; routing and the token
mapping must agree exactly, every float output to fp64 rounding.  A mistake
in either write-up (a dropped term, a wrong index or sign, a transposed
weight) shows up as a disagreement.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import moe_oracle_ref as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "route_hand_T8E4k2.json")

# (T, d, f, E, k, S, renorm, seed, logit kind)
CASES = [
    (60, 16, 24, 6, 2, 1, 0, 40, "normal"),
    (64, 32, 16, 8, 3, 0, 1, 41, "normal"),
    (50, 16, 32, 4, 4, 2, 0, 42, "normal"),      # E = k: every expert holds every token
    (90, 16, 16, 12, 5, 1, 1, 43, "ties"),       # integer logits with signed zeros
    (40, 16, 16, 7, 2, 0, 0, 44, "empty"),       # an expert nobody picks
]


def _inputs(T, d, f, E, k, S, seed, kind):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    if kind == "ties":
        z = torch.randint(-2, 3, (T, E), generator=g).float()
        z[torch.rand(T, E, generator=g) < 0.2] = -0.0
    else:
        z = torch.randn(T, E, generator=g).float()
    if kind == "empty":
        z[:, E - 1] = -30.0
    W1 = (0.1 * torch.randn(E + S, f, d, generator=g)).to(torch.bfloat16)
    W3 = (0.1 * torch.randn(E + S, f, d, generator=g)).to(torch.bfloat16)
    W2 = (0.1 * torch.randn(E + S, d, f, generator=g)).to(torch.bfloat16)
    dy = torch.randn(T, d, generator=g).to(torch.bfloat16)
    return x, z, W1, W3, W2, dy


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[0]}_E{c[3]}_k{c[4]}_S{c[5]}_r{c[6]}_{c[8]}")
def test_cpp_reference_agrees_with_numpy_oracle(case):
    T, d, f, E, k, S, renorm, seed, kind = case
    x, z, W1, W3, W2, dy = _inputs(T, d, f, E, k, S, seed, kind)
    fw = O.layer_fwd(x, z, W1, W3, W2, k=k, S=S, renorm=renorm)
    bw = O.layer_bwd(fw, dy, x, W1, W3, W2, renorm=renorm)
    sel, w, p = C.route(z.numpy(), k, renorm)
    assert np.array_equal(sel, fw.routing.sel)
    np.testing.assert_allclose(w, fw.routing.w, rtol=1e-13, atol=0)
    np.testing.assert_allclose(p, fw.routing.p, rtol=1e-13, atol=1e-300)
    perm = C.permute(sel, E)
    for name in ("counts", "offsets", "dest", "row_token", "row_slot"):
        assert np.array_equal(perm[name], getattr(fw.perm, name)), name
    if kind == "empty":
        assert perm["counts"][E - 1] == 0
    ref = C.layer(x, z, W1, W3, W2, dy, k, S, renorm)
    want = {"y": fw.y, "dx": bw.dx, "dlogits": bw.dlogits, "dW1": bw.dW1, "dW3": bw.dW3, "dW2": bw.dW2,
            "dw": bw.dw}
    for name, v in want.items():
        scale = max(1.0, float(np.abs(v).max()))
        np.testing.assert_allclose(ref[name], v, rtol=1e-10, atol=1e-12 * scale, err_msg=name)
    if kind == "empty":
        for name in ("dW1", "dW3", "dW2"):
            assert not ref[name][E - 1].any()


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_cpp_reference_on_the_hand_case(case):
    z = np.array(case["logits"], dtype=np.float32)
    sel, w, _ = C.route(z, case["k"], 0)
    assert sel.tolist() == case["sel"]
    want_w = np.array([[eval(s, {"exp": math.exp}) for s in row] for row in case["w_renorm0_closed_form"]])
    np.testing.assert_allclose(w, want_w, rtol=1e-14)
    perm = C.permute(sel, case["E"])
    for name in ("counts", "offsets", "dest", "row_token", "row_slot"):
        assert perm[name].tolist() == case[name], name


def test_cpp_reference_rejects_non_finite_logits():
    z = np.zeros((3, 4), np.float32)
    z[1, 2] = np.nan
    with pytest.raises(ValueError):
        C.route(z, 2)

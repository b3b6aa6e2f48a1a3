"""Each kernel alone through its C-ABI entry point against the CPU oracle
(GPU).  Integer tables bit-exact; floats at the tolerances of gpu_util."""
import json
import os

import numpy as np
import pytest
import torch

from combine_fp32_softmax_gb300 import moe
from combine_fp32_softmax_gb300.configs import TINY, MoEConfig
from combine_fp32_softmax_gb300.inputs import make_layer_inputs, make_logits, make_x
from oracle import moe_oracle as O
from tests.gpu_util import (DEV, assert_bf16_rounding_close, assert_grad_close, device_error, np64,
                            to_dev)

pytestmark = pytest.mark.gpu

MID = MoEConfig("mid_T700_d256_f320_E6_k2_S1", 700, 256, 320, 6, 2, S=1)
D192 = MoEConfig("d192_T333_d192_f128_E4_k3", 333, 192, 128, 4, 3)
SKEW = MoEConfig("skew_T2048_d128_f192_E32_k4_zipf", 2048, 128, 192, 32, 4, zipf=True)
EK = MoEConfig("ek_T200_d128_f128_E4_k4_renorm", 200, 128, 128, 4, 4, renorm=1)
GEMM_CFGS = [TINY, MID, D192, SKEW, EK]


@pytest.fixture(params=["pair", "single"])
def gemm_mode(request):
    """Runs a GEMM test with every kind on CTA pairs (256-row tiles) and
    again with one CTA per 128-row tile."""
    prev = moe.moe_set_gemm_pair_kinds(moe.ALL_PAIR_KINDS if request.param == "pair" else 0)
    yield request.param
    moe.moe_set_gemm_pair_kinds(prev)


def _route(cfg, logits_dev):
    ws = moe.alloc_workspace(cfg, DEV)
    idx = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=DEV)
    w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=DEV)
    moe.moe_route(cfg, logits_dev, idx, w, ws)
    return idx, w, ws


def _dispatch(cfg, idx, x_dev, ws):
    R = cfg.T * cfg.k
    t = {n: torch.empty(s, dtype=torch.int32, device=DEV) for n, s in
         [("counts", cfg.E), ("offsets", cfg.E + 1), ("dest", R), ("row_token", R), ("row_slot", R)]}
    Xp = torch.empty(R, cfg.d, dtype=torch.bfloat16, device=DEV) if x_dev is not None else None
    moe.moe_dispatch(cfg, idx, x_dev, t["counts"], t["offsets"], t["dest"], t["row_token"], t["row_slot"], Xp, ws)
    return t, Xp


# ------------------------------------------------------------------ router
@pytest.mark.parametrize("cfg", [TINY, MID, SKEW, EK,
                                 MoEConfig("e256k8", 1000, 64, 64, 256, 8),
                                 MoEConfig("e1k1", 77, 64, 64, 1, 1),
                                 MoEConfig("e33k5_renorm", 513, 64, 64, 33, 5, renorm=1)],
                         ids=lambda c: c.name)
def test_route_matches_oracle(cfg):
    z = make_logits(cfg, seed=1)
    idx, w, ws = _route(cfg, z.to(DEV))
    ref = O.route(z, cfg.k, cfg.renorm)
    assert np.array_equal(idx.cpu().numpy(), ref.sel)
    np.testing.assert_allclose(np64(w), ref.w, rtol=4e-6, atol=0)
    assert device_error(ws) == (0, 0)


def test_route_ties_and_signed_zero():
    """Integer-valued logits with many ties and signed zeros."""
    cfg = MoEConfig("ties", 4096, 64, 64, 48, 6)
    g = torch.Generator().manual_seed(7)
    z = torch.randint(-2, 3, (cfg.T, cfg.E), generator=g).float()
    z[torch.rand(cfg.T, cfg.E, generator=g) < 0.2] = -0.0
    idx, w, ws = _route(cfg, z.to(DEV))
    ref = O.route(z, cfg.k)
    assert np.array_equal(idx.cpu().numpy(), ref.sel)
    np.testing.assert_allclose(np64(w), ref.w, rtol=4e-6)


@pytest.mark.parametrize("E,k", [(20, 3), (48, 6), (200, 8)])
def test_route_extreme_and_tied_values(E, k):
    """Logits drawn from a small set of extreme and tied values (+-FLT_MAX,
    the smallest denormals, the smallest normal, signed zeros, +-1): the
    picks follow (value desc, index asc) exactly, with -0.0 == +0.0 and
    denormals ordered by value, through the router and through the fused
    routing of the layer forward."""
    cfg = MoEConfig(f"extreme_E{E}_k{k}", 1500, 64, 64, E, k)
    tiny = np.finfo(np.float32).tiny
    fmax = np.finfo(np.float32).max
    dmin = np.float32(1e-45)
    vals = np.array([fmax, -fmax, dmin, -dmin, 2 * dmin, tiny, -tiny, 0.0, -0.0, 1.0, -1.0, 1.0, 0.0],
                    dtype=np.float32)
    rng = np.random.default_rng(E)
    z = torch.from_numpy(vals[rng.integers(0, len(vals), size=(cfg.T, E))].copy())
    z[: cfg.T // 2][z[: cfg.T // 2] == fmax] = 1.0  # half the rows without the saturating value
    idx, w, ws = _route(cfg, z.to(DEV))
    ref = O.route(z, cfg.k)
    assert np.array_equal(idx.cpu().numpy(), ref.sel)
    np.testing.assert_allclose(np64(w), ref.w, rtol=4e-6, atol=0)
    assert device_error(ws) == (0, 0)
    g = {"logits": z.to(DEV), "x": torch.zeros(cfg.T, cfg.d, dtype=torch.bfloat16, device=DEV),
         "W1": torch.zeros(E, cfg.f, cfg.d, dtype=torch.bfloat16, device=DEV),
         "W3": torch.zeros(E, cfg.f, cfg.d, dtype=torch.bfloat16, device=DEV),
         "W2": torch.zeros(E, cfg.d, cfg.f, dtype=torch.bfloat16, device=DEV)}
    ws2 = moe.alloc_workspace(cfg, DEV)
    y = torch.empty(cfg.T, cfg.d, dtype=torch.float32, device=DEV)
    idx2 = torch.empty_like(idx)
    w2 = torch.empty_like(w)
    moe.moe_layer_fwd(cfg, g["logits"], g["x"], g["W1"], g["W3"], g["W2"], y, idx2, w2, ws2)
    assert device_error(ws2) == (0, 0)
    assert torch.equal(idx2, idx) and torch.equal(w2, w)
    perm = O.permute(ref.sel, E)
    for name in ("counts", "offsets", "dest", "row_token", "row_slot"):
        assert np.array_equal(moe.ws_view(ws2, cfg, name).cpu().numpy(), getattr(perm, name)), name


def test_hand_case_through_the_library():
    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "route_hand_T8E4k2.json")))["cases"]
    for case in cases:
        z = torch.tensor(case["logits"], dtype=torch.float32)
        cfg = MoEConfig("hand", z.shape[0], 64, 64, case["E"], case["k"])
        idx, w, ws = _route(cfg, z.to(DEV))
        assert idx.cpu().tolist() == case["sel"]
        t, _ = _dispatch(cfg, idx, None, ws)
        for name in ("counts", "offsets", "dest", "row_token", "row_slot"):
            assert t[name].cpu().tolist() == case[name], name


def test_nonfinite_logit_is_reported():
    cfg = MoEConfig("nan", 300, 64, 64, 8, 2)
    z = make_logits(cfg)
    z[123, 5] = float("nan")
    idx, w, ws = _route(cfg, z.to(DEV))
    code, info = device_error(ws)
    assert code == moe.MOE_ERR_NONFINITE and info == 123
    # the tables stay a valid permutation
    t, _ = _dispatch(cfg, idx, None, ws)
    assert sorted(t["dest"].cpu().tolist()) == list(range(cfg.T * cfg.k))


# ------------------------------------------------------------ permutation
@pytest.mark.parametrize("cfg", [TINY, MID, SKEW, EK, MoEConfig("big_e", 70000, 64, 64, 200, 8)],
                         ids=lambda c: c.name)
def test_dispatch_tables_bit_exact(cfg):
    inp_x = make_x(cfg, seed=2)
    z = make_logits(cfg, seed=2)
    idx, w, ws = _route(cfg, z.to(DEV))
    x_dev = inp_x.to(DEV)
    t, Xp = _dispatch(cfg, idx, x_dev, ws)
    ref = O.permute(O.route(z, cfg.k).sel, cfg.E)
    for name in ("counts", "offsets", "dest", "row_token", "row_slot"):
        assert np.array_equal(t[name].cpu().numpy(), getattr(ref, name)), name
    assert torch.equal(Xp, x_dev[t["row_token"].long()])


def test_dispatch_rejects_out_of_range_expert_index():
    cfg = MoEConfig("badidx", 100, 64, 64, 8, 2)
    idx = torch.zeros(cfg.T, cfg.k, dtype=torch.int32)
    idx[:, 1] = 1
    idx[17, 0] = 9  # out of range
    ws = moe.alloc_workspace(cfg, DEV)
    t, _ = _dispatch(cfg, idx.to(DEV), None, ws)
    code, info = device_error(ws)
    assert code == moe.MOE_ERR_ARG and info == 17 * 2
    assert sorted(t["dest"].cpu().tolist()) == list(range(cfg.T * cfg.k))


# ---------------------------------------------------------------- combine
@pytest.mark.parametrize("cfg", [TINY, MID, EK], ids=lambda c: c.name)
def test_combine_and_dispatch_bwd_sum_in_slot_order(cfg):
    """y[t] = ((O'[dest[t,0]] + O'[dest[t,1]]) + ...) + shared rows, in fp32:
    the same sum in the same order in numpy float32 gives the same bits."""
    z = make_logits(cfg, seed=3)
    idx, _, ws = _route(cfg, z.to(DEV))
    t, _ = _dispatch(cfg, idx, None, ws)
    g = torch.Generator().manual_seed(3)
    Op = torch.randn(cfg.Rs, cfg.d, generator=g, dtype=torch.float32)
    dest = t["dest"].cpu().numpy().reshape(cfg.T, cfg.k)
    Opn = Op.numpy()
    want = Opn[dest[:, 0]].copy()
    for j in range(1, cfg.k):
        want = want + Opn[dest[:, j]]
    for s in range(cfg.S):
        want = want + Opn[cfg.R + s * cfg.T: cfg.R + (s + 1) * cfg.T]
    for fn in (moe.moe_combine, moe.moe_dispatch_bwd):
        y = torch.empty(cfg.T, cfg.d, dtype=torch.float32, device=DEV)
        fn(cfg, Op.to(DEV), t["dest"], y, ws)
        assert np.array_equal(y.cpu().numpy(), want)


# --------------------------------------------------------------- route bwd
@pytest.mark.parametrize("cfg", [MID, EK, MoEConfig("e64k6", 999, 64, 64, 64, 6)], ids=lambda c: c.name)
def test_route_bwd_matches_oracle(cfg):
    z = make_logits(cfg, seed=4)
    idx, w, ws = _route(cfg, z.to(DEV))
    dw = torch.randn(cfg.T, cfg.k, generator=torch.Generator().manual_seed(4))
    dz = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=DEV)
    moe.moe_route_bwd(cfg, z.to(DEV), idx, w, dw.to(DEV), dz, ws)
    ref = O.route_bwd(O.route(z, cfg.k, cfg.renorm), dw.double().numpy(), cfg.renorm)
    assert_grad_close("dlogits", dz, ref)


# ------------------------------------------------------------ expert GEMMs
def _fwd_pieces(cfg, seed=5):
    inp = make_layer_inputs(cfg, seed)
    g = to_dev(inp)
    idx, w, ws = _route(cfg, g["logits"])
    t, Xp = _dispatch(cfg, idx, g["x"], ws)
    Hw = torch.empty(cfg.Rs, cfg.f, dtype=torch.bfloat16, device=DEV)
    AB = torch.empty(cfg.Rs, 2 * cfg.f, dtype=torch.bfloat16, device=DEV)
    Op = torch.empty(cfg.Rs, cfg.d, dtype=torch.float32, device=DEV)
    moe.moe_group_gemm_swiglu(cfg, Xp, g["x"], t["offsets"], t["row_slot"], w, g["W1"], g["W3"], g["W2"],
                              Hw, AB, Op, ws)
    fw = O.layer_fwd(inp.x, inp.logits, inp.W1, inp.W3, inp.W2, k=cfg.k, S=cfg.S, renorm=cfg.renorm)
    return inp, g, idx, w, ws, t, Xp, Hw, AB, Op, fw


@pytest.mark.parametrize("cfg", GEMM_CFGS, ids=lambda c: c.name)
def test_gemm_fwd_matches_oracle(cfg, gemm_mode):
    inp, g, idx, w, ws, t, Xp, Hw, AB, Op, fw = _fwd_pieces(cfg)
    assert device_error(ws) == (0, 0)
    assert_bf16_rounding_close("a", AB[:, :cfg.f], fw.a)
    assert_bf16_rounding_close("b", AB[:, cfg.f:], fw.b)
    wrow = np.ones(cfg.Rs)
    wrow[:cfg.R] = fw.routing.w.reshape(-1)[fw.perm.row_slot]
    # Hw = bf16(w * h): one bf16 rounding of the routing-weighted activation
    assert_bf16_rounding_close("Hw", Hw, wrow[:, None] * fw.h)
    assert_grad_close("O'", Op, wrow[:, None] * fw.o)


@pytest.mark.parametrize("cfg", GEMM_CFGS, ids=lambda c: c.name)
def test_gemm_bwd_matches_oracle(cfg, gemm_mode):
    inp, g, idx, w, ws, t, Xp, Hw, AB, Op, fw = _fwd_pieces(cfg)
    bw = O.layer_bwd(fw, inp.dy, inp.x, inp.W1, inp.W3, inp.W2, renorm=cfg.renorm)
    G = torch.empty(cfg.R, cfg.d, dtype=torch.bfloat16, device=DEV)
    moe.moe_combine_bwd(cfg, g["dy"], t["row_token"], G, ws)
    assert torch.equal(G, g["dy"][t["row_token"].long()])
    nexp = cfg.E + cfg.S
    dAB = torch.empty(cfg.Rs, 2 * cfg.f, dtype=torch.bfloat16, device=DEV)
    dw = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=DEV)
    dXp = torch.empty(cfg.Rs, cfg.d, dtype=torch.float32, device=DEV)
    dW1 = torch.full((nexp, cfg.f, cfg.d), float("nan"), device=DEV)
    dW3 = torch.full((nexp, cfg.f, cfg.d), float("nan"), device=DEV)
    dW2 = torch.full((nexp, cfg.d, cfg.f), float("nan"), device=DEV)
    moe.moe_group_gemm_swiglu_bwd(cfg, G, g["dy"], Xp, g["x"], t["offsets"], t["row_slot"], t["dest"], w,
                                  g["W1"], g["W3"], g["W2"], Hw, AB, dAB, dw, dXp, dW1, dW3, dW2, 3, ws)
    assert device_error(ws) == (0, 0)
    assert_grad_close("dA", dAB[:, :cfg.f], bw.dA)
    assert_grad_close("dB", dAB[:, cfg.f:], bw.dB)
    assert_grad_close("dw", dw, bw.dw)
    assert_grad_close("dXp", dXp, bw.dXp)
    assert_grad_close("dW1", dW1, bw.dW1)
    assert_grad_close("dW3", dW3, bw.dW3)
    assert_grad_close("dW2", dW2, bw.dW2)
    counts = t["counts"].cpu().numpy()
    for e in np.nonzero(counts == 0)[0]:  # empty experts: exact zeros
        assert torch.count_nonzero(dW1[e]) == 0 and torch.count_nonzero(dW3[e]) == 0
        assert torch.count_nonzero(dW2[e]) == 0

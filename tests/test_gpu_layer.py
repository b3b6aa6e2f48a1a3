"""The whole layer (forward + backward) through moe_layer_fwd/moe_layer_bwd
against the CPU oracle, determinism, and the full-size sampled check (GPU)."""
import hashlib

import numpy as np
import pytest
import torch

from combine_fp32_softmax_gb300 import moe
from combine_fp32_softmax_gb300.configs import DSV2_LITE, LONG128K, MIXTRAL, SKEWED, TINY, MoEConfig
from combine_fp32_softmax_gb300.inputs import make_layer_inputs
from oracle import moe_oracle as O
from tests.gpu_util import (DEV, assert_grad_close, assert_layer_close, device_error, empty_outputs, np64,
                            run_layer, to_dev)

pytestmark = pytest.mark.gpu

MID = MoEConfig("mid_T700_d256_f320_E6_k2_S1", 700, 256, 320, 6, 2, S=1)
SKEW = MoEConfig("skew_T2048_d128_f192_E32_k4_zipf", 2048, 128, 192, 32, 4, zipf=True)
EK = MoEConfig("ek_T200_d128_f128_E4_k4_renorm", 200, 128, 128, 4, 4, renorm=1)
WIDE = MoEConfig("wide_T1500_d512_f704_E8_k2_S2", 1500, 512, 704, 8, 2, S=2)
# the most rows a token sums: k = 8 routed slots and S = 4 shared experts
MAXROWS = MoEConfig("maxrows_T300_d128_f192_E16_k8_S4", 300, 128, 192, 16, 8, S=4)
# the most segments a grouped GEMM walks: E = 256 routed experts (many empty) + 4 shared
MAXSEG = MoEConfig("maxseg_T400_d64_f64_E256_k8_S4", 400, 64, 64, 256, 8, S=4)
# the degenerate router: one expert, k = 1 (every token to expert 0, weight 1)
ONE = MoEConfig("one_T100_d64_f64_E1_k1", 100, 64, 64, 1, 1)
LAYER_CFGS = [TINY, MID, SKEW, EK, WIDE, MAXROWS, MAXSEG, ONE]


def _check_layer(cfg, out, inp):
    fw = O.layer_fwd(inp.x, inp.logits, inp.W1, inp.W3, inp.W2, k=cfg.k, S=cfg.S, renorm=cfg.renorm)
    bw = O.layer_bwd(fw, inp.dy, inp.x, inp.W1, inp.W3, inp.W2, renorm=cfg.renorm)
    assert np.array_equal(out["topk_idx"].cpu().numpy(), fw.routing.sel)
    np.testing.assert_allclose(np64(out["topk_w"]), fw.routing.w, rtol=4e-6)
    assert_layer_close("y", out["y"], fw.y)
    assert_grad_close("dx", out["dx"], bw.dx)
    assert_grad_close("dlogits", out["dlogits"], bw.dlogits)
    assert_grad_close("dW1", out["dW1"], bw.dW1)
    assert_grad_close("dW3", out["dW3"], bw.dW3)
    assert_grad_close("dW2", out["dW2"], bw.dW2)


@pytest.mark.parametrize("cfg", LAYER_CFGS, ids=lambda c: c.name)
def test_layer_matches_oracle(cfg):
    inp = make_layer_inputs(cfg, seed=11)
    out, ws = run_layer(cfg, to_dev(inp), fill=float("nan"))
    assert device_error(ws) == (0, 0)
    _check_layer(cfg, out, inp)


def _digest(out):
    h = hashlib.sha256()
    for k in sorted(out):
        h.update(out[k].contiguous().cpu().numpy().tobytes())
    return h.hexdigest()


def test_bitwise_identical_across_10_runs():
    cfg = MID
    g = to_dev(make_layer_inputs(cfg, seed=12))
    digests = {_digest(run_layer(cfg, g)[0]) for _ in range(10)}
    assert len(digests) == 1


def _sched_words_clear(ws, cfg):
    """The routing grid barrier's arrival count and every grouped-GEMM kind's
    tile-ticket counter and finished-CTA count are back at 0."""
    err = moe.ws_view(ws, cfg, "err").cpu().numpy()
    # six kinds' words, then the interleaved backward GEMMs' pair
    return err[8] == 0 and not err[16:16 + 2 * (len(moe.GEMM_KINDS) + 1)].any()


def test_results_do_not_depend_on_grid_size():
    """Any CTA cap (one CTA, an odd count, all SMs) gives the same bits: every
    output element has one producer and one reduction order, whether its tile
    came from the static round-robin or the ticket counter.  The scheduling
    counters are back at 0 after every call."""
    cfg = SKEW
    g = to_dev(make_layer_inputs(cfg, seed=13))
    digests = set()
    try:
        for n in (1, 7, 0):
            moe.moe_set_grid_limit(n)
            out, ws = run_layer(cfg, g)
            digests.add(_digest(out))
            assert device_error(ws) == (0, 0)
            assert _sched_words_clear(ws, cfg)
    finally:
        moe.moe_set_grid_limit(0)
    assert len(digests) == 1


def test_cuda_graph_replay_gives_the_same_bits():
    """The layer's forward and backward captured in one CUDA graph (the
    cooperative routing launch, CTA-pair launches, the fork/join of the
    weight-gradient stream) and replayed several times give the bits of the
    plain calls, with the scheduling counters back at 0 after each replay."""
    cfg = MID
    g = to_dev(make_layer_inputs(cfg, seed=24))
    ref, _ = run_layer(cfg, g)
    ws = moe.alloc_workspace(cfg, DEV)
    out = empty_outputs(cfg)
    run_layer(cfg, g, ws=ws, out=out)  # first launches outside the capture (attributes, tensor maps)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        run_layer(cfg, g, ws=ws, out=out)
    for _ in range(3):
        for t in out.values():
            if t.dtype.is_floating_point:
                t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert device_error(ws) == (0, 0)
        assert _sched_words_clear(ws, cfg)
        for k in ref:
            assert torch.equal(out[k], ref[k]), k


def test_weight_gradient_tickets_reset_between_launches():
    """Many back-to-back weight-gradient launches (the W part alone, on the B
    part's dA|dB and Hw kept in the workspace; both tile shapes) keep giving
    the same bits: each launch starts from a ticket counter that the previous
    one's last CTA set back to 0."""
    cfg = MID
    g = to_dev(make_layer_inputs(cfg, seed=23))
    ref, ws = run_layer(cfg, g)
    prev = moe.moe_set_gemm_pair_kinds(moe.ALL_PAIR_KINDS)
    try:
        for mask in (moe.ALL_PAIR_KINDS, 0, moe.ALL_PAIR_KINDS):
            moe.moe_set_gemm_pair_kinds(mask)
            for _ in range(4):
                out = empty_outputs(cfg)
                moe.moe_layer_bwd(cfg, g["dy"], g["logits"], g["x"], g["W1"], g["W3"], g["W2"], ref["topk_idx"],
                                  ref["topk_w"], ws, out["dx"], out["dlogits"], out["dW1"], out["dW3"], out["dW2"],
                                  which=2)
                assert device_error(ws) == (0, 0)
                assert _sched_words_clear(ws, cfg)
                for k in ("dW1", "dW3", "dW2"):
                    assert torch.equal(out[k], ref[k]), (mask, k)
    finally:
        moe.moe_set_gemm_pair_kinds(prev)


@pytest.mark.parametrize("cfg", LAYER_CFGS, ids=lambda c: c.name)
def test_cta_pair_tiles_equal_single_cta_tiles_bitwise(cfg):
    """Every grouped GEMM on CTA pairs (256-row tiles, tcgen05 CTA group of
    two) gives the same bits as one CTA per 128-row tile: each output element
    is the same fp32 sum over K in the same order.  The configurations cover
    segments that end inside the pair's first half (an odd CTA with no valid
    row) and weight-gradient row counts that are not multiples of 256."""
    g = to_dev(make_layer_inputs(cfg, seed=18))
    prev = moe.moe_set_gemm_pair_kinds(0)
    try:
        a, wsa = run_layer(cfg, g)
        moe.moe_set_gemm_pair_kinds(moe.ALL_PAIR_KINDS)
        b, wsb = run_layer(cfg, g, fill=float("nan"))
    finally:
        moe.moe_set_gemm_pair_kinds(prev)
    assert device_error(wsa) == (0, 0) and device_error(wsb) == (0, 0)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    for name in ("Hw", "AB", "Op", "dAB"):
        assert torch.equal(moe.ws_view(wsa, cfg, name), moe.ws_view(wsb, cfg, name)), name


def _gemm_settings():
    mask = moe.moe_set_gemm_pair_kinds(moe.ALL_PAIR_KINDS)
    moe.moe_set_gemm_pair_kinds(mask)
    depths, stages, orders, epis = [], [], [], []
    for k in range(len(moe.GEMM_KINDS)):
        depths.append(moe.moe_set_gemm_prefetch(k, 0))
        moe.moe_set_gemm_prefetch(k, depths[-1])
        stages.append(moe.moe_set_gemm_stages(k, 0))
        moe.moe_set_gemm_stages(k, stages[-1])
    for k in (4, 5):
        orders.append(moe.moe_set_gemm_tile_order(k, 0))
        moe.moe_set_gemm_tile_order(k, orders[-1])
    for k in FP32_KINDS:
        epis.append(moe.moe_set_gemm_epilogue(k, 0))
        moe.moe_set_gemm_epilogue(k, epis[-1])
    return mask, depths, stages, orders, epis


FP32_KINDS = (1, 3, 4, 5)  # GEMM 2, dX, dW1/dW3, dW2: fp32 outputs


def _restore_gemm_settings(saved):
    mask, depths, stages, orders, epis = saved
    for k, e in zip(FP32_KINDS, epis):
        moe.moe_set_gemm_epilogue(k, e)
    moe.moe_set_gemm_pair_kinds(mask)
    for k, d in enumerate(depths):
        moe.moe_set_gemm_prefetch(k, d)
    for k, n in enumerate(stages):
        moe.moe_set_gemm_stages(k, n)
    for k, o in zip((4, 5), orders):
        moe.moe_set_gemm_tile_order(k, o)


@pytest.mark.parametrize("depth", [4, 16])
def test_next_tile_l2_prefetch_keeps_bits(depth):
    """Prefetching the next tile's K blocks into L2 only moves data earlier."""
    cfg = WIDE
    g = to_dev(make_layer_inputs(cfg, seed=20))
    saved = _gemm_settings()
    try:
        a, _ = run_layer(cfg, g)
        for k in range(len(moe.GEMM_KINDS)):
            moe.moe_set_gemm_prefetch(k, depth)
        b, wsb = run_layer(cfg, g, fill=float("nan"))
    finally:
        _restore_gemm_settings(saved)
    assert device_error(wsb) == (0, 0)
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("cfg", [MID, SKEW], ids=lambda c: c.name)
def test_autotune_chooses_per_kind_and_keeps_bits(cfg):
    """The measured autotuner returns a valid choice for every grouped-GEMM
    kind (tile shape, prefetch depth, tile order, stages) and the forward and
    backward variant, applies the GEMM choices, and the layer's outputs
    afterwards are the same bits as the oracle-checked defaults'."""
    g = to_dev(make_layer_inputs(cfg, seed=19))
    saved = _gemm_settings()
    try:
        ref, ws = run_layer(cfg, g)
        ref = {k: v.clone() for k, v in ref.items()}
        o = empty_outputs(cfg)
        res = moe.moe_autotune(cfg, g["logits"], g["x"], g["W1"], g["W3"], g["W2"], g["dy"], o["y"], o["topk_idx"],
                               o["topk_w"], o["dx"], o["dlogits"], o["dW1"], o["dW3"], o["dW2"], ws)
        kinds = res["kinds"]
        assert set(kinds) == set(moe.GEMM_KINDS)
        for i, (name, c) in enumerate(kinds.items()):
            top = moe.moe_gemm_max_stages(i, 2 if c["pair"] else 1)
            assert c["pair"] in (0, 1) and c["prefetch_kb"] in (0, 4, 8) and c["us"] > 0, (name, c)
            assert c["tile_order"] in ((0, 1) if i >= 4 else (0,)) and top - 1 <= c["stages"] <= top, (name, c)
        assert res["fwd_megakernel"] in (0, 1) and res["bwd_megakernel"] in (0, 1)
        assert min(res["fwd_us"] + res["bwd_us"]) > 0, res
        mask, depths, stages, orders, epis = _gemm_settings()
        assert epis == [kinds[moe.GEMM_KINDS[k]]["epi_direct"] for k in FP32_KINDS]
        assert mask == sum(kinds[n]["pair"] << i for i, n in enumerate(moe.GEMM_KINDS))
        assert depths == [kinds[n]["prefetch_kb"] for n in moe.GEMM_KINDS]
        assert orders == [kinds["dw13"]["tile_order"], kinds["dw2"]["tile_order"]]
        tuned, ws2 = run_layer(cfg, g, fill=float("nan"))
    finally:
        _restore_gemm_settings(saved)
    assert device_error(ws2) == (0, 0)
    for k in ref:
        assert torch.equal(ref[k], tuned[k]), k


@pytest.mark.parametrize("cfg", LAYER_CFGS, ids=lambda c: c.name)
def test_tile_order_stage_count_and_epilogue_stores_keep_bits(cfg):
    """The interleaved weight-gradient tile order, fewer pipeline stages (one
    less than fits, and two) and the direct (unstaged) epilogue stores of the
    fp32-output kinds, on both tile shapes, give the same bits: they change
    which CTA computes a tile, when, and how its results travel to memory,
    never the arithmetic.  The shapes include partial last tiles of every
    kind, so the direct stores' row and column limits are exercised."""
    g = to_dev(make_layer_inputs(cfg, seed=25))
    saved = _gemm_settings()
    try:
        ref, ref_ws = run_layer(cfg, g)
        ref = {k: v.clone() for k, v in ref.items()}
        for mask in (moe.ALL_PAIR_KINDS, 0):
            moe.moe_set_gemm_pair_kinds(mask)
            for order, stages, epi in ((1, 0, 0), (0, -1, 1), (1, 2, 1), (0, 0, 1)):
                for k in (4, 5):
                    moe.moe_set_gemm_tile_order(k, order)
                for k in FP32_KINDS:
                    moe.moe_set_gemm_epilogue(k, epi)
                for k in range(len(moe.GEMM_KINDS)):
                    top = moe.moe_gemm_max_stages(k, 2 if mask else 1)
                    moe.moe_set_gemm_stages(k, top - 1 if stages < 0 else stages)
                out, ws = run_layer(cfg, g, fill=float("nan"))
                assert device_error(ws) == (0, 0)
                for k in ref:
                    assert torch.equal(ref[k], out[k]), (mask, order, stages, epi, k)
                for name in ("Op", "dXp"):
                    assert torch.equal(moe.ws_view(ws, cfg, name), moe.ws_view(ref_ws, cfg, name)), name
    finally:
        _restore_gemm_settings(saved)


@pytest.mark.parametrize("cfg", [MID, SKEW], ids=lambda c: c.name)
def test_bw_overlap_on_a_second_stream_keeps_bits(cfg):
    """The weight-gradient GEMMs on the library's second stream (forked after
    dH, joined before return) give the same bits as the single-stream order,
    and the caller's stream alone orders the results."""
    g = to_dev(make_layer_inputs(cfg, seed=21))
    prev = moe.moe_set_bwd_overlap(False)
    try:
        a, _ = run_layer(cfg, g)
        moe.moe_set_bwd_overlap(True)
        b, wsb = run_layer(cfg, g, fill=float("nan"))
        c = {k: v.clone() for k, v in b.items()}  # read right after the call, ordered by the stream only
    finally:
        moe.moe_set_bwd_overlap(prev)
    assert device_error(wsb) == (0, 0)
    for k in a:
        assert torch.equal(a[k], c[k]), k


def test_b_and_w_parts_split():
    """which=1 then which=2 gives the same bits as which=3."""
    cfg = MID
    g = to_dev(make_layer_inputs(cfg, seed=14))
    full, _ = run_layer(cfg, g, which=3)
    ws = moe.alloc_workspace(cfg, DEV)
    part, ws = run_layer(cfg, g, ws=ws, which=1)
    moe.moe_layer_bwd(cfg, g["dy"], g["logits"], g["x"], g["W1"], g["W3"], g["W2"], part["topk_idx"],
                      part["topk_w"], ws, None, None, part["dW1"], part["dW3"], part["dW2"], which=2)
    for k in full:
        assert torch.equal(full[k], part[k]), k


@pytest.mark.parametrize("cfg", LAYER_CFGS, ids=lambda c: c.name)
def test_interleaved_backward_gemms_equal_separate_launches(cfg):
    """dX, dW1/dW3 and dW2 as one launch with interleaved tiles (both tile
    shapes) give the bits of the separate launches: every output, dXp, and
    the scheduling words back at 0."""
    g = to_dev(make_layer_inputs(cfg, seed=26))
    ref, ref_ws = run_layer(cfg, g)
    ref = {k: v.clone() for k, v in ref.items()}
    prev = moe.moe_set_bwd_fused_gemms(True)
    saved = moe.moe_set_gemm_pair_kinds(moe.ALL_PAIR_KINDS)
    try:
        for mask in (moe.ALL_PAIR_KINDS, 0):
            moe.moe_set_gemm_pair_kinds(mask)
            out, ws = run_layer(cfg, g, fill=float("nan"))
            assert device_error(ws) == (0, 0)
            assert _sched_words_clear(ws, cfg)
            for k in ref:
                assert torch.equal(ref[k], out[k]), (mask, k)
            assert torch.equal(moe.ws_view(ws, cfg, "dXp"), moe.ws_view(ref_ws, cfg, "dXp"))
    finally:
        moe.moe_set_bwd_fused_gemms(bool(prev))
        moe.moe_set_gemm_pair_kinds(saved)


def test_interleaved_backward_gemms_do_not_depend_on_grid_size():
    cfg = SKEW
    g = to_dev(make_layer_inputs(cfg, seed=27))
    ref = _digest(run_layer(cfg, g)[0])
    prev = moe.moe_set_bwd_fused_gemms(True)
    try:
        for n in (1, 7, 0):
            moe.moe_set_grid_limit(n)
            out, ws = run_layer(cfg, g)
            assert device_error(ws) == (0, 0) and _sched_words_clear(ws, cfg)
            assert _digest(out) == ref, n
    finally:
        moe.moe_set_grid_limit(0)
        moe.moe_set_bwd_fused_gemms(bool(prev))


@pytest.mark.parametrize("cfg", LAYER_CFGS, ids=lambda c: c.name)
def test_megakernel_bitwise_equals_kernel_chain(cfg):
    """The single-launch forward equals the unfused kernel chain bit for bit
    (every output and every activation saved for the backward)."""
    g = to_dev(make_layer_inputs(cfg, seed=15))
    a, wsa = run_layer(cfg, g, use_megakernel=0)
    b, wsb = run_layer(cfg, g, use_megakernel=1, fill=float("nan"))
    assert device_error(wsb) == (0, 0)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    for name in ("Xp", "Hw", "AB", "Op"):
        assert torch.equal(moe.ws_view(wsa, cfg, name), moe.ws_view(wsb, cfg, name)), name


def test_megakernel_does_not_depend_on_grid_size():
    cfg = WIDE
    g = to_dev(make_layer_inputs(cfg, seed=16))
    ref = _digest(run_layer(cfg, g, use_megakernel=0)[0])
    try:
        for n in (1, 7, 0):
            moe.moe_set_grid_limit(n)
            assert _digest(run_layer(cfg, g, use_megakernel=1)[0]) == ref, n
    finally:
        moe.moe_set_grid_limit(0)


def test_megakernel_wait_timeout_is_reported_and_context_survives():
    """A task that never completes (set on the host) makes its dependants'
    bounded waits run out: the kernel returns MOE_ERR_TIMEOUT through the
    device error word, and the next launches on the same context work."""
    cfg = MID
    g = to_dev(make_layer_inputs(cfg, seed=17))
    first_gemm1_ticket = -(-cfg.R // 32)  # gather tasks come first, 32 rows each
    ws = moe.alloc_workspace(cfg, DEV)
    out = {k: v for k, v in run_layer(cfg, g, ws=ws, use_megakernel=0)[0].items()}
    try:
        moe.moe_debug_skip_megakernel_task(first_gemm1_ticket)
        moe.moe_layer_fwd(cfg, g["logits"], g["x"], g["W1"], g["W3"], g["W2"], out["y"], out["topk_idx"],
                          out["topk_w"], ws, use_megakernel=1)
        code, info = device_error(ws)
    finally:
        moe.moe_debug_skip_megakernel_task(-1)
    assert code == moe.MOE_ERR_TIMEOUT, (code, info)
    ref, _ = run_layer(cfg, g, use_megakernel=0)
    again, ws2 = run_layer(cfg, g, use_megakernel=1)
    assert device_error(ws2) == (0, 0)
    for k in ref:
        assert torch.equal(ref[k], again[k]), k


TABLES = ("counts", "offsets", "dest", "row_token", "row_slot")
# ragged T, one expert row per lane (E = 32), the wider rows (E = 100, 256),
# a single histogram block (T = 8) and a single token (T = 1, one CTA)
ROUTE_CFGS = [TINY, MID, SKEW, EK, MoEConfig("e100_T1234_d64_f64_E100_k5", 1234, 64, 64, 100, 5),
              MoEConfig("e256_T333_d64_f64_E256_k8_renorm", 333, 64, 64, 256, 8, renorm=1),
              MoEConfig("t8_d64_f64_E4_k2", 8, 64, 64, 4, 2),
              MoEConfig("t1_d64_f64_E5_k3_S1", 1, 64, 64, 5, 3, S=1)]


def _fwd_tables(cfg, g, fused, grid):
    prev = moe.moe_set_route_fusion(fused)
    moe.moe_set_grid_limit(grid)
    try:
        ws = moe.alloc_workspace(cfg, DEV)
        out = empty_outputs(cfg)
        moe.moe_layer_fwd(cfg, g["logits"], g["x"], g["W1"], g["W3"], g["W2"], out["y"], out["topk_idx"],
                          out["topk_w"], ws)
        assert device_error(ws) == (0, 0)
        res = {name: moe.ws_view(ws, cfg, name).clone() for name in TABLES}
        res.update(topk_idx=out["topk_idx"], topk_w=out["topk_w"], y=out["y"])
        return res
    finally:
        moe.moe_set_route_fusion(prev)
        moe.moe_set_grid_limit(0)


@pytest.mark.parametrize("cfg", ROUTE_CFGS, ids=lambda c: c.name)
def test_fused_routing_tables_equal_three_kernels_and_oracle(cfg):
    """The cooperative route + histogram + scan + scatter launch gives the
    tables of the three separate kernels bit for bit, on any grid (one CTA
    walks every histogram block and every expert row), and they are the
    oracle's permutation."""
    inp = make_layer_inputs(cfg, seed=21)
    g = to_dev(inp)
    ref = _fwd_tables(cfg, g, fused=0, grid=0)
    for grid in (0, 1, 3):
        got = _fwd_tables(cfg, g, fused=1, grid=grid)
        for name in ref:
            assert torch.equal(got[name], ref[name]), (grid, name)
    routing = O.route(inp.logits, cfg.k, cfg.renorm)
    perm = O.permute(routing.sel, cfg.E)
    assert np.array_equal(ref["topk_idx"].cpu().numpy(), routing.sel)
    for name in TABLES:
        assert np.array_equal(ref[name].cpu().numpy(), getattr(perm, name)), name


def test_fused_routing_barrier_timeout_is_reported_and_context_survives():
    """A grid barrier whose arrival count is poisoned on the host (no CTA is
    ever the last to arrive) runs out its bounded wait: the launch returns
    with MOE_ERR_TIMEOUT in the device error word instead of hanging, and
    after moe_ws_init the same workspace routes correctly again."""
    cfg = MID
    g = to_dev(make_layer_inputs(cfg, seed=22))
    ref = _fwd_tables(cfg, g, fused=0, grid=0)
    ws = moe.alloc_workspace(cfg, DEV)
    out = empty_outputs(cfg)
    moe.ws_view(ws, cfg, "err")[8] = -5
    moe.moe_layer_fwd(cfg, g["logits"], g["x"], g["W1"], g["W3"], g["W2"], out["y"], out["topk_idx"],
                      out["topk_w"], ws)
    code, info = device_error(ws)
    assert code == moe.MOE_ERR_TIMEOUT and info == 1, (code, info)
    moe.moe_ws_init(cfg, ws)
    moe.moe_layer_fwd(cfg, g["logits"], g["x"], g["W1"], g["W3"], g["W2"], out["y"], out["topk_idx"],
                      out["topk_w"], ws)
    assert device_error(ws) == (0, 0)
    for name in TABLES:
        assert torch.equal(moe.ws_view(ws, cfg, name), ref[name]), name
    assert torch.equal(out["y"], ref["y"])


BWD_MK = 3 | moe.MOE_BWD_MEGAKERNEL


@pytest.mark.parametrize("cfg", LAYER_CFGS, ids=lambda c: c.name)
def test_bwd_megakernel_bitwise_equals_kernel_chain(cfg):
    """The backward input part as one MegaKernel launch (gather, dH, dX, dx
    sum) equals the kernel chain bit for bit: every output and every
    activation it leaves in the workspace."""
    g = to_dev(make_layer_inputs(cfg, seed=22))
    a, wsa = run_layer(cfg, g, which=3)
    b, wsb = run_layer(cfg, g, which=BWD_MK, fill=float("nan"))
    assert device_error(wsb) == (0, 0)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    for name in ("G", "dAB", "dXp", "dw"):
        assert torch.equal(moe.ws_view(wsa, cfg, name), moe.ws_view(wsb, cfg, name)), name


def test_bwd_megakernel_does_not_depend_on_grid_size():
    cfg = WIDE
    g = to_dev(make_layer_inputs(cfg, seed=23))
    ref = _digest(run_layer(cfg, g, which=3)[0])
    try:
        for n in (1, 7, 0):
            moe.moe_set_grid_limit(n)
            assert _digest(run_layer(cfg, g, which=BWD_MK)[0]) == ref, n
    finally:
        moe.moe_set_grid_limit(0)


def test_bwd_megakernel_wait_timeout_is_reported_and_context_survives():
    """A dH task that never completes (set on the host): the dX tasks of its
    row block and the dx sums wait, run out of time, and the kernel returns
    MOE_ERR_TIMEOUT; the next launches on the same context work."""
    cfg = MID
    g = to_dev(make_layer_inputs(cfg, seed=24))
    first_dh_ticket = -(-cfg.R // 32)  # gather tasks come first, 32 rows each
    out, ws = run_layer(cfg, g)
    try:
        moe.moe_debug_skip_megakernel_task(first_dh_ticket)
        moe.moe_layer_bwd(cfg, g["dy"], g["logits"], g["x"], g["W1"], g["W3"], g["W2"], out["topk_idx"],
                          out["topk_w"], ws, out["dx"], out["dlogits"], out["dW1"], out["dW3"], out["dW2"],
                          which=BWD_MK)
        code, info = device_error(ws)
    finally:
        moe.moe_debug_skip_megakernel_task(-1)
    assert code == moe.MOE_ERR_TIMEOUT, (code, info)
    ref, _ = run_layer(cfg, g, which=3)
    again, ws2 = run_layer(cfg, g, which=BWD_MK)
    assert device_error(ws2) == (0, 0)
    for k in ref:
        assert torch.equal(ref[k], again[k]), k


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [DSV2_LITE, MIXTRAL, SKEWED, LONG128K], ids=lambda c: c.name)
def test_full_size_sampled_parity(cfg):
    """Every workload at full size, in the benchmark's launch configuration:
    routing and the permutation in full, y / dx / dlogits on 2048 seeded
    tokens, and 352 weight-gradient entries of each of dW1, dW3 and dW2 for
    several experts (largest, smallest, a middle one, one more, the shared
    ones; 4224 entries or more), each summed over the expert's whole segment;
    empty experts' gradients exactly 0."""
    inp = make_layer_inputs(cfg, seed=0)
    out, ws = run_layer(cfg, to_dev(inp))
    assert device_error(ws) == (0, 0)
    routing = O.route(inp.logits, cfg.k, cfg.renorm)
    assert np.array_equal(out["topk_idx"].cpu().numpy(), routing.sel)
    perm = O.permute(routing.sel, cfg.E)
    for name in ("counts", "offsets", "dest", "row_token", "row_slot"):
        assert np.array_equal(moe.ws_view(ws, cfg, name).cpu().numpy(), getattr(perm, name)), name
    rng = np.random.default_rng(0)
    ntok = 2048
    toks = np.sort(rng.choice(cfg.T, ntok, replace=False))
    _, y, dx, dz, _ = O.tokens_fwd_bwd(inp.x, inp.logits.numpy(), inp.W1, inp.W3, inp.W2, inp.dy, cfg.k, cfg.S,
                                       cfg.renorm, toks)
    assert_layer_close("y", np64(out["y"])[toks], y)
    assert_grad_close("dx", np64(out["dx"])[toks], dx)
    assert_grad_close("dlogits", np64(out["dlogits"])[toks], dz)
    counts = perm.counts
    nonempty = np.nonzero(counts)[0]
    experts = [int(np.argmax(counts)), int(nonempty[np.argmin(counts[nonempty])]), int(nonempty[len(nonempty) // 2])]
    others = [int(e) for e in nonempty if int(e) not in experts]
    experts += [others[int(rng.integers(0, len(others)))]] if others else []
    experts += [cfg.E + s for s in range(cfg.S)]
    for e in np.nonzero(counts == 0)[0][:4]:  # empty experts: exact zeros
        for gpu in (out["dW1"], out["dW3"], out["dW2"]):
            assert torch.count_nonzero(gpu[int(e)]) == 0
    for which, gpu in (("W1", out["dW1"]), ("W3", out["dW3"]), ("W2", out["dW2"])):
        for e in experts:
            nr, nc = gpu.shape[1], gpu.shape[2]
            # 22 hidden units x 16 entries each (the oracle forms one
            # segment-long column per hidden unit)
            nf = nr if which in ("W1", "W3") else nc
            units = np.repeat(rng.choice(nf, 22, replace=False), 16)
            if which in ("W1", "W3"):
                rows, cols = units, rng.integers(0, nc, units.size)
            else:
                rows, cols = rng.integers(0, nr, units.size), units
            ref = O.dW_entries(inp.x, inp.logits.numpy(), inp.W1, inp.W3, inp.W2, inp.dy, cfg.k, cfg.S,
                               cfg.renorm, which, e, rows, cols, routing=routing, perm=perm)
            got = np64(gpu[e])[rows, cols]
            if counts[e] == 0 if e < cfg.E else False:
                assert np.all(got == 0)
                continue
            assert_grad_close(f"d{which}[{e}] sample", got, ref)

"""Run-to-run bitwise determinism at full size, in the configurations the
benchmark uses.

The layer must give the same bits on every run (UniEP page, section 2.2,
Algorithm 1: a token-to-expert mapping that does not depend on execution
order, so the backward is bit-level consistent).  The small-shape tests
cover the mechanisms one at a time; these run the paths that only the full
workloads reach: 76 CTA pairs on every grouped GEMM, the weight-gradient
tiles drawn from the ticket counter (longest segments first, 176 long
shared-expert tiles at the DeepSeek-V2-Lite-like shape), the backward's
weight-gradient GEMMs on the second stream, the cooperative routing launch
on every SM, and CUDA-graph replay of the whole step.

Every comparison is exact (torch.equal on the device) over every output
(y, dx, dlogits, dW1, dW3, dW2, topk_idx, topk_w) and the activations the
forward saves for the backward.
"""
import pytest
import torch

from combine_fp32_softmax_gb300 import moe
from combine_fp32_softmax_gb300.configs import DSV2_LITE, LONG128K
from combine_fp32_softmax_gb300.inputs import make_layer_inputs
from tests.gpu_util import check_guards, device_error, empty_outputs, guarded_workspace, run_layer, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAVED = ("Xp", "Hw", "AB", "Op", "G", "dAB", "dXp", "dw")


def _snapshot(out, ws, cfg):
    snap = {k: v.clone() for k, v in out.items()}
    for name in SAVED:
        snap["ws." + name] = moe.ws_view(ws, cfg, name).clone()
    return snap


def _same(a, b):
    """Names of the tensors whose bits differ."""
    return [k for k in a if not torch.equal(a[k], b[k])]


def _poison(out):
    for t in out.values():
        if t.dtype.is_floating_point:
            t.fill_(float("nan"))
        else:
            t.fill_(-1)


@pytest.fixture(scope="module")
def bench_layer():
    """The benchmark workload with the library's defaults (CTA pairs on every
    kind, B/W overlap on, fused routing), run once as the reference."""
    cfg = DSV2_LITE
    saved = (moe.moe_set_gemm_pair_kinds(moe.ALL_PAIR_KINDS), moe.moe_set_bwd_overlap(True),
             moe.moe_set_route_fusion(True))
    moe.moe_set_grid_limit(0)
    g = to_dev(make_layer_inputs(cfg, seed=0))
    ws = guarded_workspace(cfg)
    out = empty_outputs(cfg)
    run_layer(cfg, g, ws=ws, out=out)
    assert device_error(ws) == (0, 0)
    ref = _snapshot(out, ws, cfg)
    yield cfg, g, ws, out, ref
    moe.moe_set_gemm_pair_kinds(saved[0])
    moe.moe_set_bwd_overlap(bool(saved[1]))
    moe.moe_set_route_fusion(bool(saved[2]))


def test_bench_workload_10_graph_replays_bitwise_identical(bench_layer):
    """Ten replays of the captured step (how bench.py times it), each into
    poisoned outputs, give the reference bits."""
    cfg, g, ws, out, ref = bench_layer
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        run_layer(cfg, g, ws=ws, out=out)
    for i in range(10):
        _poison(out)
        graph.replay()
        torch.cuda.synchronize()
        assert device_error(ws) == (0, 0), i
        diff = _same(ref, _snapshot(out, ws, cfg))
        assert not diff, (i, diff)


def test_bench_workload_10_plain_runs_bitwise_identical(bench_layer):
    """Ten host-launched runs, each on a fresh workspace and poisoned
    outputs, give the reference bits."""
    cfg, g, _, _, ref = bench_layer
    for i in range(10):
        ws = guarded_workspace(cfg)
        out = empty_outputs(cfg)
        run_layer(cfg, g, ws=ws, out=out, fill=float("nan"))
        assert device_error(ws) == (0, 0), i
        diff = _same(ref, _snapshot(out, ws, cfg))
        assert not diff, (i, diff)
        del ws, out
        check_guards()


def test_bench_workload_grid_size_does_not_change_bits(bench_layer):
    """Seven CTAs (three pairs and a lone CTA for the single-CTA launches)
    instead of every SM: each tile meets other tiles on its CTA, the ticket
    counter hands out the weight-gradient tiles in another interleaving, and
    the bits stay the same."""
    cfg, g, _, _, ref = bench_layer
    try:
        moe.moe_set_grid_limit(7)
        ws = guarded_workspace(cfg)
        out = empty_outputs(cfg)
        run_layer(cfg, g, ws=ws, out=out, fill=float("nan"))
        assert device_error(ws) == (0, 0)
        diff = _same(ref, _snapshot(out, ws, cfg))
    finally:
        moe.moe_set_grid_limit(0)
    assert not diff, diff


def test_bench_workload_megakernels_equal_the_chain(bench_layer):
    """The forward MegaKernel and the backward input-part MegaKernel at full
    size give the chain's bits (the tests at small shapes check this on
    eight layer shapes)."""
    cfg, g, _, _, ref = bench_layer
    ws = guarded_workspace(cfg)
    out = empty_outputs(cfg)
    run_layer(cfg, g, ws=ws, out=out, use_megakernel=1, which=3 | moe.MOE_BWD_MEGAKERNEL, fill=float("nan"))
    assert device_error(ws) == (0, 0)
    diff = _same(ref, _snapshot(out, ws, cfg))
    assert not diff, diff


def test_long_sequence_3_runs_bitwise_identical():
    """The 128k-token layer (1,048,576 GEMM rows, 786,432 routed) three times,
    each on a fresh workspace and poisoned outputs: the same bits."""
    cfg = LONG128K
    g = to_dev(make_layer_inputs(cfg, seed=0))
    ref = None
    for i in range(3):
        ws = guarded_workspace(cfg)
        out = empty_outputs(cfg)
        run_layer(cfg, g, ws=ws, out=out, fill=float("nan"))
        assert device_error(ws) == (0, 0), i
        snap = {k: v.clone() for k, v in out.items()} if ref is None else out
        if ref is None:
            ref = snap
        else:
            diff = _same(ref, snap)
            assert not diff, (i, diff)
        del ws, out
        check_guards()
        torch.cuda.empty_cache()

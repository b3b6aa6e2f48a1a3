"""The debug build's checks (compiled in with -DMOE_DEBUG): a bad index in
a caller-given table is recorded in the device error word as MOE_ERR_ARG
with the site and the token (or row) it was found at, and the access it
guards is skipped or clamped -- never made.  These tests run only against
the debug build (tests/test_gpu_debug_build.py runs them in a child process
with MOE_GB300_DEBUG_LIB=1); the release build compiles the checks out.

Every bad value here stays inside what the release build already tolerates
(clamped or skipped indices, a segment table whose end the kernels do not
read), so no launch touches memory outside its buffers either way."""
import os

import pytest
import torch

from combine_fp32_softmax_gb300 import moe
from combine_fp32_softmax_gb300.configs import MoEConfig
from combine_fp32_softmax_gb300.inputs import make_layer_inputs
from tests.gpu_util import DEV, guarded_workspace, run_layer, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(os.environ.get("MOE_GB300_DEBUG_LIB") != "1", reason="debug build only")]

CFG = MoEConfig("dbg_T300_d128_f128_E8_k2_S1", 300, 128, 128, 8, 2, S=1)
SITE = {"gather": 0x41, "scatter": 0x42, "sum": 0x43, "segments": 0x50}


def _layer():
    g = to_dev(make_layer_inputs(CFG, seed=5))
    out, ws = run_layer(CFG, g)
    assert moe.moe_get_device_error(ws) == (0, 0)
    return g, out, ws


def _fresh_ws():
    return guarded_workspace(CFG)


def test_combine_reports_a_row_outside_the_gemm_rows():
    _, _, ws = _layer()
    dest = moe.ws_view(ws, CFG, "dest").clone()
    dest[2 * CFG.k + 1] = CFG.Rs + 7  # token 2, slot 1
    y = torch.empty(CFG.T, CFG.d, dtype=torch.float32, device=DEV)
    w2 = _fresh_ws()
    moe.moe_combine(CFG, moe.ws_view(ws, CFG, "Op"), dest, y, w2)
    assert moe.moe_get_device_error(w2) == (moe.MOE_ERR_ARG, SITE["sum"] << 24 | 2)


def test_combine_bwd_reports_a_token_outside_the_batch():
    g, _, ws = _layer()
    row_token = moe.ws_view(ws, CFG, "row_token").clone()
    row_token[9] = CFG.T + 1
    G = torch.empty(CFG.R, CFG.d, dtype=torch.bfloat16, device=DEV)
    w2 = _fresh_ws()
    moe.moe_combine_bwd(CFG, g["dy"], row_token, G, w2)
    assert moe.moe_get_device_error(w2) == (moe.MOE_ERR_ARG, SITE["gather"] << 24 | 9)
    assert torch.count_nonzero(G[9]) == 0  # the bad row is written as zeros, nothing is read for it


def test_grouped_gemm_reports_a_segment_table_not_ending_at_R():
    g, out, ws = _layer()
    offsets = moe.ws_view(ws, CFG, "offsets").clone()
    offsets[CFG.E] = CFG.R - 1  # the last entry is not read by the kernels, only checked
    Hw = torch.empty(CFG.Rs, CFG.f, dtype=torch.bfloat16, device=DEV)
    Op = torch.empty(CFG.Rs, CFG.d, dtype=torch.float32, device=DEV)
    w2 = _fresh_ws()
    moe.moe_group_gemm_swiglu(CFG, moe.ws_view(ws, CFG, "Xp"), g["x"], offsets, moe.ws_view(ws, CFG, "row_slot"),
                              out["topk_w"], g["W1"], g["W3"], g["W2"], Hw, None, Op, w2)
    code, info = moe.moe_get_device_error(w2)
    assert code == moe.MOE_ERR_ARG and (info >> 24) == SITE["segments"], (code, hex(info))
    # the rows themselves are computed as without the check
    ref = moe.ws_view(ws, CFG, "Op")
    assert torch.equal(Op, ref)

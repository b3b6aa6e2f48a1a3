"""moe_dispatch_noalloc, the entry point for callers that cannot provide a
workspace (e.g. an operator registered with a zero-byte workspace, or code
whose device memory a host framework planned in advance, so nothing may
allocate while it runs).  It must give exactly the tables and gathered rows
that moe_dispatch gives, call after call, although it keeps its scratch in
one array inside the library that every call reuses.  This file is named to
be collected last so a failure here never hides the other tests."""
import ctypes

import pytest
import torch

from combine_fp32_softmax_gb300 import moe
from combine_fp32_softmax_gb300.configs import MoEConfig
from combine_fp32_softmax_gb300.inputs import make_logits, make_x

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
NAMES = ("counts", "offsets", "dest", "row_token", "row_slot")


def _tables(cfg):
    R = cfg.T * cfg.k
    t = {n: torch.full((s,), -7, dtype=torch.int32, device=DEV) for n, s in
         [("counts", cfg.E), ("offsets", cfg.E + 1), ("dest", R), ("row_token", R), ("row_slot", R)]}
    t["Xp"] = torch.zeros(R, cfg.d, dtype=torch.bfloat16, device=DEV)
    return t


def _route(cfg, seed):
    ws = moe.alloc_workspace(cfg, DEV)
    idx = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=DEV)
    w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=DEV)
    moe.moe_route(cfg, make_logits(cfg, seed).to(DEV), idx, w, ws)
    return idx, ws


def _noalloc(cfg, idx, x, t):
    """Direct call through the C ABI (no workspace argument exists)."""
    lib = moe.lib()
    c = moe.cfg_of(cfg)
    p = lambda v: ctypes.c_void_p(v.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.moe_dispatch_noalloc(ctypes.byref(c), p(idx), p(x), p(t["counts"]), p(t["offsets"]), p(t["dest"]),
                                    p(t["row_token"]), p(t["row_slot"]), p(t["Xp"]), stream)


def test_noalloc_dispatch_matches_moe_dispatch_twice_in_a_row():
    # two calls in a row with different shapes: the second reuses the array
    # the first left behind, so stale scratch would show up here
    for cfg, seed in [(MoEConfig("na1", 3000, 256, 64, 64, 6), 1), (MoEConfig("na2", 777, 128, 64, 16, 3), 2)]:
        idx, ws = _route(cfg, seed)
        x = make_x(cfg, seed).to(DEV)
        want = _tables(cfg)
        moe.moe_dispatch(cfg, idx, x, want["counts"], want["offsets"], want["dest"], want["row_token"],
                         want["row_slot"], want["Xp"], ws)
        got = _tables(cfg)
        assert _noalloc(cfg, idx, x, got) == moe.MOE_OK
        torch.cuda.synchronize()
        for n in NAMES:  # integer tables: bit-exact
            assert torch.equal(got[n], want[n]), n
        assert torch.equal(got["Xp"], want["Xp"])


def test_noalloc_rejects_shapes_beyond_its_scratch():
    cfg = MoEConfig("too_big", 70000, 64, 64, 256, 8)  # 256 * ceil(70000/32) > 524,256
    idx = torch.zeros(1, dtype=torch.int32, device=DEV)
    t = {n: idx for n in NAMES}
    t["Xp"] = torch.zeros(1, dtype=torch.bfloat16, device=DEV)
    assert _noalloc(cfg, idx, t["Xp"], t) == moe.MOE_ERR_SHAPE


def test_noalloc_calls_after_the_first_leave_device_memory_unchanged():
    # the first call on the device may load the library's kernels and place
    # the scratch array; after it, calls must not change the device's free
    # memory (nothing allocated, nothing freed)
    cfg = MoEConfig("na3", 4096, 256, 64, 64, 6)
    idx, _ = _route(cfg, 3)
    x = make_x(cfg, 3).to(DEV)
    t = _tables(cfg)
    assert _noalloc(cfg, idx, x, t) == moe.MOE_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        assert _noalloc(cfg, idx, x, t) == moe.MOE_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)


def test_noalloc_clamps_out_of_range_indices_like_moe_dispatch():
    # one index past the last expert and one below 0: both entry points clamp
    # them into range and give the same tables; moe_dispatch reports the
    # first bad slot in its workspace's error word
    cfg = MoEConfig("na4", 500, 128, 64, 16, 2)
    idx, _ = _route(cfg, 4)
    flat = idx.view(-1)
    flat[37] = cfg.E
    flat[401] = -3
    x = make_x(cfg, 4).to(DEV)
    ws = moe.alloc_workspace(cfg, DEV)
    want = _tables(cfg)
    moe.moe_dispatch(cfg, idx, x, want["counts"], want["offsets"], want["dest"], want["row_token"],
                     want["row_slot"], want["Xp"], ws)
    code, info = moe.moe_get_device_error(ws)
    assert code == moe.MOE_ERR_ARG and info in (37, 401), (code, info)
    got = _tables(cfg)
    assert _noalloc(cfg, idx, x, got) == moe.MOE_OK
    torch.cuda.synchronize()
    for n in NAMES:
        assert torch.equal(got[n], want[n]), n
    assert torch.equal(got["Xp"], want["Xp"])

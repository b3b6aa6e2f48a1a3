"""The C-ABI library without a GPU: it loads, exports every function that
include/moe.h declares, and rejects bad arguments on the host before any
CUDA call (no device is touched by these tests)."""
import ctypes
import os
import re

import pytest

from combine_fp32_softmax_gb300 import build as B
from combine_fp32_softmax_gb300 import moe
from combine_fp32_softmax_gb300.configs import ALL, TINY, MoEConfig

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        B.build()
    return moe.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["moe_route", "moe_dispatch", "moe_group_gemm_swiglu", "moe_combine", "moe_layer_fwd",
                 "moe_combine_bwd", "moe_group_gemm_swiglu_bwd", "moe_dispatch_bwd", "moe_route_bwd",
                 "moe_layer_bwd", "moe_workspace_bytes", "moe_get_device_error"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def _cfg(**kw):
    base = dict(T=512, d_model=256, d_ff=512, E=8, k=2, n_shared=0, renorm=0)
    base.update(kw)
    return moe.moe_cfg(*[base[n] for n, _ in moe.moe_cfg._fields_])


@pytest.mark.parametrize("bad", [dict(E=0), dict(E=257), dict(k=9, E=16), dict(k=5, E=4), dict(d_model=96),
                                 dict(d_ff=100), dict(T=0), dict(n_shared=5), dict(renorm=2),
                                 dict(T=1 << 30, k=4)])
def test_bad_shapes_are_rejected(lib, bad):
    c = _cfg(**bad)
    assert lib.moe_workspace_bytes(ctypes.byref(c)) == 0
    fake = ctypes.c_void_p(1 << 20)
    assert lib.moe_route(ctypes.byref(c), fake, fake, fake, fake, None) == moe.MOE_ERR_SHAPE


def test_null_and_misaligned_pointers_are_rejected(lib):
    c = _cfg()
    ok = ctypes.c_void_p(1 << 20)        # never dereferenced: checks run first
    odd = ctypes.c_void_p((1 << 20) + 8)  # 8-byte aligned only
    ws_odd = ctypes.c_void_p((1 << 20) + 16)  # 16- but not 256-byte aligned
    assert lib.moe_route(ctypes.byref(c), None, ok, ok, ok, None) == moe.MOE_ERR_ARG
    assert lib.moe_route(ctypes.byref(c), odd, ok, ok, ok, None) == moe.MOE_ERR_ALIGN
    assert lib.moe_route(ctypes.byref(c), ok, ok, ok, ws_odd, None) == moe.MOE_ERR_ALIGN
    assert lib.moe_combine(ctypes.byref(c), ok, ok, None, ok, None) == moe.MOE_ERR_ARG
    assert lib.moe_layer_bwd(ctypes.byref(c), *([ok] * 14), 0, None) == moe.MOE_ERR_ARG  # which=0
    assert lib.moe_layer_bwd(ctypes.byref(c), *([ok] * 9), None, ok, ok, ok, ok, 3, None) == moe.MOE_ERR_ARG
    assert lib.moe_get_device_error(None, None, None, None) == moe.MOE_ERR_ARG


@pytest.mark.parametrize("cfg", ALL + [MoEConfig("odd", 700, 192, 320, 6, 2, S=1)], ids=lambda c: c.name)
def test_workspace_layout_matches_binding_mirror(lib, cfg):
    total = moe.moe_workspace_bytes(cfg)
    offs = moe.ws_offsets(cfg)
    assert total >= offs["_mk"] + 64
    assert total % 256 == 0
    # every region is 256-byte aligned (TMA needs 16)
    assert all(v % 256 == 0 for v in offs.values())


def test_gemm_knobs_reject_bad_kinds_and_values(lib):
    # tile order: weight-gradient kinds (4, 5) only, order 0 or 1
    for kind in (0, 1, 2, 3, 6, -1):
        assert lib.moe_set_gemm_tile_order(kind, 1) == moe.MOE_ERR_ARG
    assert lib.moe_set_gemm_tile_order(4, 2) == moe.MOE_ERR_ARG
    # epilogue stores: fp32-output kinds (1, 3, 4, 5) only, 0 or 1
    for kind in (0, 2, 6, -1):
        assert lib.moe_set_gemm_epilogue(kind, 1) == moe.MOE_ERR_ARG
    assert lib.moe_set_gemm_epilogue(3, 7) == moe.MOE_ERR_ARG
    # stages: known kinds, non-negative
    assert lib.moe_set_gemm_stages(6, 3) == moe.MOE_ERR_ARG
    assert lib.moe_set_gemm_stages(0, -1) == moe.MOE_ERR_ARG
    assert lib.moe_gemm_max_stages(9, 1) == 0 and lib.moe_gemm_max_stages(0, 3) == 0


def test_gemm_knobs_round_trip_and_stage_limits(lib):
    """Each setter returns the previous value; the stage limits are those of
    the shared-memory ring (one CTA per tile: 48 KB stages, CTA pairs: 32 KB).
    Direct epilogue stores free the staging memory for a seventh stage on
    pairs; a 48 KB stage does not fit in it."""
    assert [lib.moe_gemm_max_stages(k, 1) for k in range(6)] == [4] * 6
    assert [lib.moe_gemm_max_stages(k, 2) for k in range(6)] == [6] * 6
    for kind in (1, 3, 4, 5):
        prev = lib.moe_set_gemm_epilogue(kind, 1)
        assert lib.moe_gemm_max_stages(kind, 2) == 7 and lib.moe_gemm_max_stages(kind, 1) == 4
        lib.moe_set_gemm_epilogue(kind, prev)
        assert lib.moe_gemm_max_stages(kind, 2) == 6
    for kind in (4, 5):
        prev = lib.moe_set_gemm_tile_order(kind, 1)
        assert lib.moe_set_gemm_tile_order(kind, prev) == 1
    for kind in (1, 3, 4, 5):
        prev = lib.moe_set_gemm_epilogue(kind, 1)
        assert lib.moe_set_gemm_epilogue(kind, prev) == 1
    for kind in range(6):
        prev = lib.moe_set_gemm_stages(kind, 3)
        assert lib.moe_set_gemm_stages(kind, prev) == 3


def test_rank_bases_rejects_bad_arguments(lib):
    ok = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert lib.moe_rank_bases(ok, 2, 8, ok, 2, ok, None, None) == moe.MOE_ERR_SHAPE   # rank >= G
    assert lib.moe_rank_bases(ok, 0, 8, ok, 0, ok, None, None) == moe.MOE_ERR_SHAPE   # G = 0
    assert lib.moe_rank_bases(ok, 2, 257, ok, 0, ok, None, None) == moe.MOE_ERR_SHAPE  # E > 256
    assert lib.moe_rank_bases(None, 2, 8, ok, 0, ok, None, None) == moe.MOE_ERR_ARG
    assert lib.moe_rank_bases(ok, 2, 8, ok, 0, None, None, None) == moe.MOE_ERR_ARG
    assert lib.moe_rank_bases(odd, 2, 8, ok, 0, ok, None, None) == moe.MOE_ERR_ALIGN
    assert lib.moe_rank_bases(ok, 2, 8, ok, 0, ok, odd, None) == moe.MOE_ERR_ALIGN

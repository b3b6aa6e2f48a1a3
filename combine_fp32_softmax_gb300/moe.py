"""Python binding of libmoe_gb300 (include/moe.h).

Argument marshalling only: every function turns torch CUDA tensors into raw
device pointers and the current CUDA stream, calls the C entry point of the
same name, and raises MoeError on a non-zero status.  All arithmetic runs in
the library's CUDA kernels; there is no fallback path.  If the library is
not built, loading it raises immediately.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import DEBUG_LIB_PATH, LIB_PATH
from .configs import MoEConfig

CODES = {0: "MOE_OK", -1: "MOE_ERR_ARG", -2: "MOE_ERR_SHAPE", -3: "MOE_ERR_ALIGN",
         -4: "MOE_ERR_CUDA", -5: "MOE_ERR_NONFINITE", -6: "MOE_ERR_TIMEOUT"}
MOE_OK, MOE_ERR_ARG, MOE_ERR_SHAPE, MOE_ERR_ALIGN = 0, -1, -2, -3
MOE_ERR_CUDA, MOE_ERR_NONFINITE, MOE_ERR_TIMEOUT = -4, -5, -6


class MoeError(RuntimeError):
    def __init__(self, name: str, code: int):
        super().__init__(f"{name} returned {code} ({CODES.get(code, '?')})")
        self.code = code


class moe_tune_result(ctypes.Structure):
    _fields_ = [("pair", ctypes.c_int * 6), ("prefetch_kb", ctypes.c_int * 6), ("us", ctypes.c_float * 6),
                ("tile_order", ctypes.c_int * 6), ("stages", ctypes.c_int * 6), ("epi_direct", ctypes.c_int * 6),
                ("fwd_megakernel", ctypes.c_int),
                ("bwd_megakernel", ctypes.c_int), ("fwd_us", ctypes.c_float * 2), ("bwd_us", ctypes.c_float * 2)]


class moe_cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("T", "d_model", "d_ff", "E", "k", "n_shared", "renorm")]


def cfg_of(c: MoEConfig) -> moe_cfg:
    return moe_cfg(c.T, c.d, c.f, c.E, c.k, c.S, c.renorm)


_P = ctypes.c_void_p
_I = ctypes.c_int
_CFG = ctypes.POINTER(moe_cfg)
# name -> argument types (after the cfg pointer, before ws/stream where present)
_SIGS = {
    "moe_workspace_bytes": ([_CFG], ctypes.c_size_t),
    "moe_ws_init": ([_CFG, _P, _P], _I),
    "moe_route": ([_CFG, _P, _P, _P, _P, _P], _I),
    "moe_dispatch": ([_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_token_addresses": ([_CFG] + [_P] * 7, _I),
    "moe_rank_bases": ([_P, _I, _I, _P, _I, _P, _P, _P], _I),
    "moe_dispatch_noalloc": ([_CFG] + [_P] * 9, _I),
    "moe_group_gemm_swiglu": ([_CFG] + [_P] * 13, _I),
    "moe_combine": ([_CFG, _P, _P, _P, _P, _P], _I),
    "moe_layer_fwd": ([_CFG] + [_P] * 9 + [_I, _P], _I),
    "moe_combine_bwd": ([_CFG, _P, _P, _P, _P, _P], _I),
    "moe_group_gemm_swiglu_bwd": ([_CFG] + [_P] * 19 + [_I, _P, _P], _I),
    "moe_dispatch_bwd": ([_CFG, _P, _P, _P, _P, _P], _I),
    "moe_route_bwd": ([_CFG, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_layer_bwd": ([_CFG] + [_P] * 14 + [_I, _P], _I),
    "moe_get_device_error": ([_P, _P, ctypes.POINTER(_I), ctypes.POINTER(_I)], _I),
    "moe_num_sms": ([], _I),
    "moe_set_grid_limit": ([_I], _I),
    "moe_set_gemm_pair_kinds": ([_I], _I),
    "moe_gemm_pair_capacity": ([_I], _I),
    "moe_set_gemm_prefetch": ([_I, _I], _I),
    "moe_set_gemm_tile_order": ([_I, _I], _I),
    "moe_set_gemm_stages": ([_I, _I], _I),
    "moe_set_gemm_epilogue": ([_I, _I], _I),
    "moe_gemm_max_stages": ([_I, _I], _I),
    "moe_set_bwd_overlap": ([_I], _I),
    "moe_set_route_fusion": ([_I], _I),
    "moe_set_bwd_fused_gemms": ([_I], _I),
    "moe_autotune": ([_CFG] + [_P] * 15 + [_I, _P, ctypes.POINTER(moe_tune_result)], _I),
    "moe_debug_skip_megakernel_task": ([_I], _I),
    "moe_debug_megakernel_trace": ([_P, _I], _I),
    "moe_trace_enable": ([_I], _I),
    "moe_trace_reset": ([], _I),
    "moe_trace_read": ([_I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I)], _I),
    "moe_trace_kind_name": ([_I], ctypes.c_char_p),
}

# kernel kinds of the timing trace (MOE_K_* in include/moe.h)
TRACE_KINDS = ["route", "hist", "scan", "scatter", "gather", "gemm1_swiglu", "gemm2_scale", "combine",
               "combine_bwd", "gemm_dh", "dw_reduce", "route_bwd", "gemm_dx", "dispatch_bwd", "gemm_dw13",
               "gemm_dw2", "megakernel", "megakernel_bwd",
               "route_tables", "bwd_gemms"]

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        # MOE_GB300_DEBUG_LIB=1 loads the debug build (tests only)
        path = DEBUG_LIB_PATH if os.environ.get("MOE_GB300_DEBUG_LIB") == "1" else LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib = handle
    return _lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != 0:
        raise MoeError(name, rc)


def _cfg(c):
    return ctypes.byref(c if isinstance(c, moe_cfg) else cfg_of(c))


# ------------------------------------------------------------ entry points
def moe_workspace_bytes(cfg) -> int:
    return int(lib().moe_workspace_bytes(_cfg(cfg)))


def moe_ws_init(cfg, ws, stream=None):
    _call("moe_ws_init", _cfg(cfg), _ptr(ws), _stream(stream))


def moe_route(cfg, logits, topk_idx, topk_w, ws, stream=None):
    _call("moe_route", _cfg(cfg), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(ws), _stream(stream))


def moe_dispatch(cfg, topk_idx, x, counts, offsets, dest, row_token, row_slot, Xp, ws, stream=None):
    _call("moe_dispatch", _cfg(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets), _ptr(dest),
          _ptr(row_token), _ptr(row_slot), _ptr(Xp), _ptr(ws), _stream(stream))


def moe_dispatch_noalloc(cfg, topk_idx, x, counts, offsets, dest, row_token, row_slot, Xp, stream=None):
    _call("moe_dispatch_noalloc", _cfg(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets), _ptr(dest),
          _ptr(row_token), _ptr(row_slot), _ptr(Xp), _stream(stream))


def moe_token_addresses(cfg, topk_idx, rank_base, counts, offsets, dest, ws, stream=None):
    _call("moe_token_addresses", _cfg(cfg), _ptr(topk_idx), _ptr(rank_base), _ptr(counts), _ptr(offsets),
          _ptr(dest), _ptr(ws), _stream(stream))


def moe_rank_bases(all_counts, owner, rank, rank_base, recv_rows=None, stream=None):
    """all_counts [G, E] int32, owner [E] int32 -> rank_base [E] int32 (and recv_rows [G] int32)."""
    G, E = all_counts.shape
    _call("moe_rank_bases", _ptr(all_counts), int(G), int(E), _ptr(owner), int(rank), _ptr(rank_base),
          _ptr(recv_rows), _stream(stream))


def moe_group_gemm_swiglu(cfg, Xp, x, offsets, row_slot, topk_w, W1, W3, W2, Hw, AB, Oprime, ws, stream=None):
    _call("moe_group_gemm_swiglu", _cfg(cfg), _ptr(Xp), _ptr(x), _ptr(offsets), _ptr(row_slot), _ptr(topk_w),
          _ptr(W1), _ptr(W3), _ptr(W2), _ptr(Hw), _ptr(AB), _ptr(Oprime), _ptr(ws), _stream(stream))


def moe_combine(cfg, Oprime, dest, y, ws, stream=None):
    _call("moe_combine", _cfg(cfg), _ptr(Oprime), _ptr(dest), _ptr(y), _ptr(ws), _stream(stream))


def moe_layer_fwd(cfg, logits, x, W1, W3, W2, y, topk_idx, topk_w, ws, use_megakernel=0, stream=None):
    _call("moe_layer_fwd", _cfg(cfg), _ptr(logits), _ptr(x), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(y),
          _ptr(topk_idx), _ptr(topk_w), _ptr(ws), int(use_megakernel), _stream(stream))


def moe_combine_bwd(cfg, dy, row_token, G, ws, stream=None):
    _call("moe_combine_bwd", _cfg(cfg), _ptr(dy), _ptr(row_token), _ptr(G), _ptr(ws), _stream(stream))


def moe_group_gemm_swiglu_bwd(cfg, G, dy, Xp, x, offsets, row_slot, dest, topk_w, W1, W3, W2, Hw, AB,
                              dAB, dw, dXp, dW1, dW3, dW2, which, ws, stream=None):
    _call("moe_group_gemm_swiglu_bwd", _cfg(cfg), _ptr(G), _ptr(dy), _ptr(Xp), _ptr(x), _ptr(offsets),
          _ptr(row_slot), _ptr(dest), _ptr(topk_w), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(Hw), _ptr(AB),
          _ptr(dAB), _ptr(dw), _ptr(dXp), _ptr(dW1), _ptr(dW3), _ptr(dW2), int(which), _ptr(ws),
          _stream(stream))


def moe_dispatch_bwd(cfg, dXp, dest, dx, ws, stream=None):
    _call("moe_dispatch_bwd", _cfg(cfg), _ptr(dXp), _ptr(dest), _ptr(dx), _ptr(ws), _stream(stream))


def moe_route_bwd(cfg, logits, topk_idx, topk_w, dw, dlogits, ws, stream=None):
    _call("moe_route_bwd", _cfg(cfg), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(dw), _ptr(dlogits),
          _ptr(ws), _stream(stream))


MOE_BWD_MEGAKERNEL = 4  # add to `which`: the B part as one MegaKernel launch


def moe_layer_bwd(cfg, dy, logits, x, W1, W3, W2, topk_idx, topk_w, ws, dx, dlogits, dW1, dW3, dW2,
                  which=3, stream=None):
    _call("moe_layer_bwd", _cfg(cfg), _ptr(dy), _ptr(logits), _ptr(x), _ptr(W1), _ptr(W3), _ptr(W2),
          _ptr(topk_idx), _ptr(topk_w), _ptr(ws), _ptr(dx), _ptr(dlogits), _ptr(dW1), _ptr(dW3), _ptr(dW2),
          int(which), _stream(stream))


def moe_get_device_error(ws, stream=None):
    code, info = _I(0), _I(0)
    _call("moe_get_device_error", _ptr(ws), _stream(stream), ctypes.byref(code), ctypes.byref(info))
    return code.value, info.value


def moe_num_sms() -> int:
    return int(lib().moe_num_sms())


def moe_set_grid_limit(n: int):
    _call("moe_set_grid_limit", int(n))


GEMM_KINDS = ("gemm1", "gemm2", "dh", "dx", "dw13", "dw2")
ALL_PAIR_KINDS = (1 << len(GEMM_KINDS)) - 1


def moe_set_gemm_pair_kinds(mask: int) -> int:
    """Bit k: grouped-GEMM kind GEMM_KINDS[k] on CTA pairs. Returns the previous mask."""
    return int(lib().moe_set_gemm_pair_kinds(int(mask)))


def moe_set_gemm_prefetch(kind: int, kblocks: int) -> int:
    """Next-tile K blocks grouped-GEMM kind `kind` prefetches into L2. Returns the previous depth."""
    r = int(lib().moe_set_gemm_prefetch(int(kind), int(kblocks)))
    if r < 0:
        raise MoeError("moe_set_gemm_prefetch", r)
    return r


def moe_autotune(cfg, logits, x, W1, W3, W2, dy, y, topk_idx, topk_w, dx, dlogits, dW1, dW3, dW2, ws,
                 reps=0, stream=None) -> dict:
    """Runs the library's measured autotuner on this layer (applying its GEMM choices process-wide) and
    returns {"kinds": {kind name: {pair, prefetch_kb, tile_order, stages, us}}, "fwd_megakernel",
    "bwd_megakernel", "fwd_us": [chain, MegaKernel], "bwd_us": [chain, MegaKernel]}."""
    res = moe_tune_result()
    _call("moe_autotune", _cfg(cfg), _ptr(logits), _ptr(x), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(dy), _ptr(y),
          _ptr(topk_idx), _ptr(topk_w), _ptr(dx), _ptr(dlogits), _ptr(dW1), _ptr(dW3), _ptr(dW2), _ptr(ws),
          int(reps), _stream(stream), ctypes.byref(res))
    kinds = {name: {"pair": res.pair[i], "prefetch_kb": res.prefetch_kb[i], "tile_order": res.tile_order[i],
                    "stages": res.stages[i], "epi_direct": res.epi_direct[i], "us": res.us[i]}
             for i, name in enumerate(GEMM_KINDS)}
    return {"kinds": kinds, "fwd_megakernel": res.fwd_megakernel, "bwd_megakernel": res.bwd_megakernel,
            "fwd_us": list(res.fwd_us), "bwd_us": list(res.bwd_us)}


def moe_set_gemm_tile_order(kind: int, order: int) -> int:
    """Tile order of a weight-gradient kind (4 or 5): 0 longest first, 1 interleaved. Returns the previous order."""
    r = int(lib().moe_set_gemm_tile_order(int(kind), int(order)))
    if r < 0:
        raise MoeError("moe_set_gemm_tile_order", r)
    return r


def moe_set_gemm_epilogue(kind: int, direct: int) -> int:
    """Epilogue stores of an fp32-output kind (1, 3, 4, 5): 0 staged (TMA), 1 direct. Returns the previous mode."""
    r = int(lib().moe_set_gemm_epilogue(int(kind), int(direct)))
    if r < 0:
        raise MoeError("moe_set_gemm_epilogue", r)
    return r


def moe_set_gemm_stages(kind: int, stages: int) -> int:
    """Pipeline stages of grouped-GEMM kind `kind` (0: as many as fit). Returns the previous request."""
    r = int(lib().moe_set_gemm_stages(int(kind), int(stages)))
    if r < 0:
        raise MoeError("moe_set_gemm_stages", r)
    return r


def moe_gemm_max_stages(kind: int, cta_group: int) -> int:
    return int(lib().moe_gemm_max_stages(int(kind), int(cta_group)))


def moe_set_bwd_overlap(on: bool) -> int:
    """Weight-gradient GEMMs of the backward on a second stream beside the dX tail. Returns the previous setting."""
    return int(lib().moe_set_bwd_overlap(int(bool(on))))


def moe_set_bwd_fused_gemms(on: bool) -> int:
    """dX, dW1/dW3 and dW2 of the layer backward as one interleaved launch. Returns the previous setting."""
    return int(lib().moe_set_bwd_fused_gemms(int(bool(on))))


def moe_set_route_fusion(on: bool) -> int:
    """Router and permutation tables of moe_layer_fwd as one cooperative launch. Returns the previous setting."""
    return int(lib().moe_set_route_fusion(int(bool(on))))


def moe_gemm_pair_capacity(kind: int) -> int:
    """CTA pairs of grouped-GEMM kind `kind` resident at once on the current device."""
    return int(lib().moe_gemm_pair_capacity(int(kind)))


def moe_debug_skip_megakernel_task(ticket: int):
    _call("moe_debug_skip_megakernel_task", int(ticket))


def moe_debug_megakernel_trace(buf, records_per_cta: int = 0):
    """buf: int64 CUDA tensor of >= grid * records_per_cta * 3 elements, or None."""
    _call("moe_debug_megakernel_trace", _ptr(buf), int(records_per_cta))


def megakernel_timeline(buf, records_per_cta: int):
    """Decodes a MegaKernel trace buffer into (cta, role, ticket, start_ns, end_ns) rows, start-sorted."""
    rec = buf.view(-1, 3).cpu().tolist()
    out = []
    for meta, t0, t1 in rec:
        if t1 <= 0 or t1 < t0:
            continue
        meta &= (1 << 64) - 1
        out.append(((meta >> 40) & 0xFFFFFF, (meta >> 32) & 0xFF, meta & 0xFFFFFFFF, t0, t1))
    return sorted(out, key=lambda r: r[3])


def moe_trace_enable(on: bool):
    _call("moe_trace_enable", int(bool(on)))


def moe_trace_reset():
    _call("moe_trace_reset")


def moe_trace_read() -> dict:
    """{kernel kind: (total device ms, launches)} since the last reset."""
    out = {}
    for i, name in enumerate(TRACE_KINDS):
        ms, n = ctypes.c_double(0), _I(0)
        _call("moe_trace_read", i, ctypes.byref(ms), ctypes.byref(n))
        if n.value:
            out[name] = (ms.value, n.value)
    return out


# ------------------------------------------------------- workspace layout
def ws_offsets(cfg: MoEConfig) -> dict:
    """Byte offsets of the workspace regions, mirroring the library's layout
    (used by tests and the benchmark to look at saved activations)."""
    T, d, f, E, k, S = cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.S
    R, Rs = T * k, T * k + S * T
    nb = -(-T // 32)
    nt = -(-f // 256)  # dw partial dots per row: one per 256-column tile
    o = 0
    out = {}

    def take(name, nbytes):
        nonlocal o
        out[name] = o
        o = (o + nbytes + 255) // 256 * 256

    for name, nbytes in [("err", 256), ("hist", 4 * E * nb), ("base", 4 * E * nb), ("counts", 4 * E),
                         ("offsets", 4 * (E + 1)), ("dest", 4 * R), ("row_token", 4 * R),
                         ("row_slot", 4 * R), ("Xp", 2 * R * d), ("AB", 4 * Rs * f), ("Hw", 2 * Rs * f),
                         ("Op", 4 * Rs * d), ("G", 2 * R * d), ("dAB", 4 * Rs * f),
                         ("dXp", 4 * Rs * d), ("partial", 4 * R * nt), ("dw", 4 * T * k)]:
        take(name, nbytes)
    out["_mk"] = o
    return out


def ws_view(ws: torch.Tensor, cfg: MoEConfig, name: str) -> torch.Tensor:
    """A typed view of one workspace region."""
    T, d, f, E, k, S = cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.S
    R, Rs = T * k, T * k + S * T
    shapes = {"err": ((64,), torch.int32), "counts": ((E,), torch.int32), "offsets": ((E + 1,), torch.int32), "dest": ((R,), torch.int32),
              "row_token": ((R,), torch.int32), "row_slot": ((R,), torch.int32),
              "Xp": ((R, d), torch.bfloat16), "AB": ((Rs, 2 * f), torch.bfloat16), "Hw": ((Rs, f), torch.bfloat16),
              "Op": ((Rs, d), torch.float32), "G": ((R, d), torch.bfloat16), "dAB": ((Rs, 2 * f), torch.bfloat16),
              "dXp": ((Rs, d), torch.float32), "dw": ((T, k), torch.float32)}
    shape, dt = shapes[name]
    off = ws_offsets(cfg)[name]
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.empty(0, dtype=dt).element_size()
    return ws[off:off + nbytes].view(dt).view(*shape)


def alloc_workspace(cfg: MoEConfig, device="cuda", stream=None) -> torch.Tensor:
    ws = torch.empty(moe_workspace_bytes(cfg), dtype=torch.uint8, device=device)
    moe_ws_init(cfg, ws, stream)
    return ws

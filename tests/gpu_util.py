"""Helpers shared by the GPU tests: device copies, the layer through the C
ABI, and the tolerance rules.

Tolerances (float outputs against the fp64 oracle):
  * layer output y: max-abs <= 2e-2 and relative Frobenius <= 5e-3 (the
    stated bar for layer outputs);
  * gradients and other fp32 outputs: relative Frobenius <= 5e-3 and
    max-abs <= 2e-2 * max(1, max|reference|).  The 2e-2 absolute bar is
    stated for the layer output (entries well below 1); gradients grow with
    the rows an expert sees (weight-gradient entries reach tens at the
    Mixtral shape), so the same bar is applied in units of the largest
    reference entry.  With bf16 tensor-core operands the worst element of a
    weight gradient sits ~11x the rms error above it (rows with large
    activations carry both large values and large rounding errors), so an
    rms-scaled bar would reject correct bf16 arithmetic;
  * stored bf16 activations (Hw = w*h, [a|b]): |got - ref| <= 2^-8 |ref| +
    1e-4 rms(ref) elementwise: one bf16 rounding of an fp32 value whose own
    error is far below a bf16 ulp;
  * routing weights: relative <= 4e-6 (fp32 softmax error bound);
  * integers: bit-exact.

Every output and workspace these helpers allocate sits between two 4 KB
guard regions filled with a fixed byte pattern; after each GPU test the
guards are checked, so a kernel that writes past either end of a buffer
fails the test that ran it (a stand-in for compute-sanitizer's memcheck,
which this machine pool does not offer).

Each tolerance check also records the error it measured (relative
Frobenius, max-abs and the bar) under the running test's id; with
MOE_MARGINS_OUT set, the session writes them to that JSON file.
"""
import math

import numpy as np
import torch

from combine_fp32_softmax_gb300 import moe
from combine_fp32_softmax_gb300.configs import MoEConfig
from combine_fp32_softmax_gb300.inputs import LayerInputs

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

# ------------------------------------------------------------ error margins
MARGINS = []  # (test id, quantity, relF, max-abs, max-abs bar)
CURRENT_TEST = {"id": ""}


def _record(name, rf, err, lim):
    MARGINS.append({"test": CURRENT_TEST["id"], "name": name, "relF": rf, "maxabs": err, "maxabs_limit": lim,
                    "relF_limit": 5e-3})


# ----------------------------------------------------------- guard regions
GUARD_BYTES = 4096
GUARD_BYTE = 0xA5
_GUARDED = []  # (backing uint8 tensor, payload bytes, label)


def guarded_empty(shape, dtype, label="buffer"):
    """An uninitialised device tensor of `shape`/`dtype` that starts 4 KB into
    a larger allocation; the 4 KB before it and everything after it (at least
    4 KB) hold GUARD_BYTE until check_guards() looks at them."""
    n = math.prod(shape) * torch.empty(0, dtype=dtype).element_size()
    back = torch.empty(2 * GUARD_BYTES + (n + 255) // 256 * 256, dtype=torch.uint8, device=DEV)
    back[:GUARD_BYTES].fill_(GUARD_BYTE)
    back[GUARD_BYTES + n:].fill_(GUARD_BYTE)
    _GUARDED.append((back, n, label))
    return back[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(*shape)


def guarded_workspace(cfg: MoEConfig):
    """moe.alloc_workspace with guard regions (the payload stays 256-byte
    aligned: the backing allocation is, and the guard is 4 KB)."""
    ws = guarded_empty((moe.moe_workspace_bytes(cfg),), torch.uint8, label="ws")
    moe.moe_ws_init(cfg, ws)
    return ws


def check_guards():
    """Raises if any guard byte of a buffer allocated since the last call
    changed; forgets those buffers."""
    bad = []
    if _GUARDED:
        torch.cuda.synchronize()
    for back, n, label in _GUARDED:
        head = back[:GUARD_BYTES]
        tail = back[GUARD_BYTES + n:]
        nh = int((head != GUARD_BYTE).sum())
        nt = int((tail != GUARD_BYTE).sum())
        if nh or nt:
            bad.append(f"{label}: {nh} bytes changed before, {nt} after")
    _GUARDED.clear()
    assert not bad, "writes outside a buffer: " + "; ".join(bad)


def np64(t) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def relf(got, ref) -> float:
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


def assert_layer_close(name, got, ref):
    got = np64(got) if torch.is_tensor(got) else got
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    rf = relf(got, ref)
    _record(name, rf, err, 2e-2)
    assert rf <= 5e-3 and err <= 2e-2, f"{name}: relF={rf:.3e} maxabs={err:.3e}"


def assert_grad_close(name, got, ref):
    got = np64(got) if torch.is_tensor(got) else got
    if ref.size == 0:
        return
    err = float(np.abs(got - ref).max())
    rf = relf(got, ref)
    lim = 2e-2 * max(1.0, float(np.abs(ref).max()))
    _record(name, rf, err, lim)
    assert rf <= 5e-3 and err <= lim, f"{name}: relF={rf:.3e} maxabs={err:.3e} (limit {lim:.3e})"


def assert_bf16_rounding_close(name, got, ref):
    got = np64(got) if torch.is_tensor(got) else got
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * rms
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{name}: {int(bad.sum())} elements beyond one bf16 rounding, worst " \
                          f"{float(np.abs(got - ref).max()):.3e}"


def to_dev(inp: LayerInputs) -> dict:
    return {k: getattr(inp, k).to(DEV).contiguous() for k in ("x", "logits", "W1", "W3", "W2", "dy")}


def empty_outputs(cfg: MoEConfig) -> dict:
    f32, i32 = torch.float32, torch.int32
    nexp = cfg.E + cfg.S
    shapes = dict(y=((cfg.T, cfg.d), f32), topk_idx=((cfg.T, cfg.k), i32), topk_w=((cfg.T, cfg.k), f32),
                  dx=((cfg.T, cfg.d), f32), dlogits=((cfg.T, cfg.E), f32), dW1=((nexp, cfg.f, cfg.d), f32),
                  dW3=((nexp, cfg.f, cfg.d), f32), dW2=((nexp, cfg.d, cfg.f), f32))
    return {k: guarded_empty(shape, dt, label=k) for k, (shape, dt) in shapes.items()}


def run_layer(cfg: MoEConfig, g: dict, ws=None, out=None, use_megakernel=0, which=3, fill=None):
    """Forward then backward through the C ABI; returns (outputs, ws)."""
    if ws is None:
        ws = guarded_workspace(cfg)
    if out is None:
        out = empty_outputs(cfg)
    if fill is not None:  # poison outputs to prove they are fully overwritten
        for t in out.values():
            if t.dtype.is_floating_point:
                t.fill_(fill)
    moe.moe_layer_fwd(cfg, g["logits"], g["x"], g["W1"], g["W3"], g["W2"], out["y"], out["topk_idx"],
                      out["topk_w"], ws, use_megakernel=use_megakernel)
    moe.moe_layer_bwd(cfg, g["dy"], g["logits"], g["x"], g["W1"], g["W3"], g["W2"], out["topk_idx"],
                      out["topk_w"], ws, out["dx"], out["dlogits"], out["dW1"], out["dW3"], out["dW2"],
                      which=which)
    return out, ws


def device_error(ws):
    torch.cuda.synchronize()
    return moe.moe_get_device_error(ws)

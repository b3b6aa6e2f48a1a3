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
  * stored bf16 activations (H, [a|b]): |got - ref| <= 2^-8 |ref| +
    1e-4 rms(ref) elementwise: one bf16 rounding of an fp32 value whose own
    error is far below a bf16 ulp;
  * routing weights: relative <= 4e-6 (fp32 softmax error bound);
  * integers: bit-exact.
"""
import numpy as np
import torch

from combine_fp32_softmax_gb300 import moe
from combine_fp32_softmax_gb300.configs import MoEConfig
from combine_fp32_softmax_gb300.inputs import LayerInputs

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def np64(t) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def relf(got, ref) -> float:
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


def assert_layer_close(name, got, ref):
    got = np64(got) if torch.is_tensor(got) else got
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    rf = relf(got, ref)
    assert rf <= 5e-3 and err <= 2e-2, f"{name}: relF={rf:.3e} maxabs={err:.3e}"


def assert_grad_close(name, got, ref):
    got = np64(got) if torch.is_tensor(got) else got
    if ref.size == 0:
        return
    err = float(np.abs(got - ref).max())
    rf = relf(got, ref)
    lim = 2e-2 * max(1.0, float(np.abs(ref).max()))
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
    return dict(
        y=torch.empty(cfg.T, cfg.d, dtype=f32, device=DEV),
        topk_idx=torch.empty(cfg.T, cfg.k, dtype=i32, device=DEV),
        topk_w=torch.empty(cfg.T, cfg.k, dtype=f32, device=DEV),
        dx=torch.empty(cfg.T, cfg.d, dtype=f32, device=DEV),
        dlogits=torch.empty(cfg.T, cfg.E, dtype=f32, device=DEV),
        dW1=torch.empty(nexp, cfg.f, cfg.d, dtype=f32, device=DEV),
        dW3=torch.empty(nexp, cfg.f, cfg.d, dtype=f32, device=DEV),
        dW2=torch.empty(nexp, cfg.d, cfg.f, dtype=f32, device=DEV),
    )


def run_layer(cfg: MoEConfig, g: dict, ws=None, out=None, use_megakernel=0, which=3, fill=None):
    """Forward then backward through the C ABI; returns (outputs, ws)."""
    if ws is None:
        ws = moe.alloc_workspace(cfg, DEV)
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

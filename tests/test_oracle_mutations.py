"""Plant plausible mistakes in the oracle (on the CPU, by monkeypatching) and
check that at least one pin of tests/test_oracle.py fails for each, so a
wrong oracle cannot pass its own pins."""
import numpy as np
import pytest
from scipy.special import expit

from oracle import moe_oracle as O
from tests import test_oracle as pins


def _wrong_topk_unstable(z, k):          # ties broken toward the higher index
    return (z.shape[1] - 1 - np.argsort(-z[:, ::-1], axis=1, kind="stable")[:, :k]).astype(np.int64)


def _wrong_topk_on_probs_descending_abs(z, k):   # picks by |z|
    return np.argsort(-np.abs(z), axis=1, kind="stable")[:, :k].astype(np.int64)


def _wrong_swiglu_swapped(xr, W1e, W3e, W2e):     # gate and up swapped
    a = xr @ W3e.T; b = xr @ W1e.T
    h = O.silu(a) * b
    return a, b, h, h @ W2e.T


def _wrong_silu(a):                        # sigmoid instead of silu
    return expit(a)


def _wrong_dsilu(a):                       # sign error inside the derivative
    s = expit(a)
    return s * (1.0 + a * s)


def _wrong_route_bwd(routing, dw, renorm):  # drops the softmax-Jacobian cross term
    T, E = routing.p.shape
    out = np.zeros((T, E))
    np.put_along_axis(out, routing.sel, dw * routing.w, axis=1)
    return out


def _wrong_permute_reversed(sel, E):       # descending token order inside a segment
    p = O._orig_permute(sel, E)
    rs = p.row_slot.copy()
    for e in range(E):
        rs[p.offsets[e]:p.offsets[e + 1]] = rs[p.offsets[e]:p.offsets[e + 1]][::-1]
    dest = np.empty_like(p.dest); dest[rs] = np.arange(len(rs))
    return O.Permutation(p.counts, p.offsets, dest, rs // sel.shape[1], rs)


MUTATIONS = {
    "topk_ties_high": ("topk_select", _wrong_topk_unstable,
                       [lambda: pins.test_topk_matches_python_sort(8, 3)]),
    "topk_abs": ("topk_select", _wrong_topk_on_probs_descending_abs,
                 [lambda: pins.test_topk_matches_python_sort(8, 3)]),
    "swiglu_swapped": ("swiglu_expert", _wrong_swiglu_swapped,
                       [pins.test_dense_swiglu_special_case]),
    "silu_is_sigmoid": ("silu", _wrong_silu, [pins.test_dense_swiglu_special_case]),
    "dsilu_sign": ("dsilu", _wrong_dsilu, [lambda: pins.test_backward_matches_autograd(0, 0)]),
    "route_bwd_no_cross_term": ("route_bwd", _wrong_route_bwd,
                                [lambda: pins.test_backward_matches_autograd(0, 0)]),
    "segment_order_reversed": ("permute", _wrong_permute_reversed,
                               [lambda: pins.test_permutation_is_library_stable_sort(37, 5, 2)]),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    attr, wrong, checks = MUTATIONS[name]
    monkeypatch.setattr(O, "_orig_permute", O.permute, raising=False)
    monkeypatch.setattr(O, attr, wrong)
    for check in checks:
        with pytest.raises(AssertionError):
            check()

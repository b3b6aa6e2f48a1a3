"""ctypes wrapper of the plain C++ fp64 reference (moe_oracle_ref.cpp).
TEST INFRASTRUCTURE: the tests use it to check the numpy oracle against a
second, independent implementation of the same definitions.  The library is
compiled here on first use (g++, OpenMP) or by ``__graft_entry__.build()``.
"""
import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle_ref.cpp")
LIB = os.path.join(HERE, "_build", "libmoe_oracle_ref.so")

_lib = None


def build() -> str:
    """Compiles the reference into oracle/_build (when older than its source)."""
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("building the C++ reference failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        _lib.ref_route.argtypes = [P, I, I, I, I, P, P, P]
        _lib.ref_permute.argtypes = [P, I, I, I, P, P, P, P, P]
        _lib.ref_layer.argtypes = [P] * 6 + [I] * 7 + [P] * 7
        for f in (_lib.ref_route, _lib.ref_permute, _lib.ref_layer):
            f.restype = I
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def bf16_bits(t) -> np.ndarray:
    """The bf16 bit patterns of a CPU torch bf16 tensor, as uint16."""
    import torch
    return t.detach().contiguous().view(torch.int16).numpy().view(np.uint16)


def route(logits: np.ndarray, k: int, renorm: int = 0):
    """(sel [T,k] int32, w [T,k] fp64, p [T,E] fp64) for fp32 logits [T,E]."""
    z = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = z.shape
    sel = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    p = np.empty((T, E), np.float64)
    if lib().ref_route(_p(z), T, E, k, renorm, _p(sel), _p(w), _p(p)) != 0:
        raise ValueError("non-finite router logit")
    return sel, w, p


def permute(sel: np.ndarray, E: int) -> dict:
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    T, k = sel.shape
    R = T * k
    out = {"counts": np.empty(E, np.int32), "offsets": np.empty(E + 1, np.int32), "dest": np.empty(R, np.int32),
           "row_token": np.empty(R, np.int32), "row_slot": np.empty(R, np.int32)}
    rc = lib().ref_permute(_p(sel), T, E, k, _p(out["counts"]), _p(out["offsets"]), _p(out["dest"]),
                           _p(out["row_token"]), _p(out["row_slot"]))
    if rc != 0:
        raise ValueError("expert index out of range")
    return out


def layer(x, logits, W1, W3, W2, dy, k: int, S: int = 0, renorm: int = 0) -> dict:
    """Forward and backward of the layer; x, W1, W3, W2, dy are CPU torch bf16
    tensors, logits fp32.  Returns fp64 numpy arrays y, dx, dlogits, dW1, dW3,
    dW2, dw."""
    xb, W1b, W3b, W2b, dyb = (bf16_bits(t) for t in (x, W1, W3, W2, dy))
    z = np.ascontiguousarray(logits.detach().cpu().numpy() if hasattr(logits, "detach") else logits,
                             dtype=np.float32)
    T, d = xb.shape
    E = z.shape[1]
    nexp, f, _ = W1b.shape
    assert nexp == E + S
    out = {"y": np.empty((T, d)), "dx": np.empty((T, d)), "dlogits": np.empty((T, E)),
           "dW1": np.empty((nexp, f, d)), "dW3": np.empty((nexp, f, d)), "dW2": np.empty((nexp, d, f)),
           "dw": np.empty((T, k))}
    rc = lib().ref_layer(_p(xb), _p(z), _p(W1b), _p(W3b), _p(W2b), _p(dyb), T, d, f, E, k, S, renorm,
                         _p(out["y"]), _p(out["dx"]), _p(out["dlogits"]), _p(out["dW1"]), _p(out["dW3"]),
                         _p(out["dW2"]), _p(out["dw"]))
    if rc != 0:
        raise ValueError("non-finite router logit")
    return out

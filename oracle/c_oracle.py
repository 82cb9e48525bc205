"""ctypes wrapper of the plain-C FP64 oracle (oracle/vce_oracle.c).

TEST INFRASTRUCTURE ONLY: a second, independent implementation of the logits
form and of the linear form's product, gradients and entropy, which the tests
compare with the NumPy oracle.  Built with gcc into oracle/_build/libvce_oracle.so.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vce_oracle.c")
LIB = os.path.join(HERE, "_build", "libvce_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC") or shutil.which("gcc") or "cc"
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + ".tmp"
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:  # no OpenMP runtime: the loops run serially
        cmd.remove("-fopenmp")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"building the C oracle failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I64, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
        lib.oracle_ce_forward.argtypes = [P, I64, I64, I64, P, D, I64, P, P, P, P]
        lib.oracle_ce_forward.restype = I64
        lib.oracle_ce_backward.argtypes = [P, I64, I64, I64, P, P, P, D, I64, P]
        lib.oracle_ce_backward.restype = None
        lib.oracle_linear_logits.argtypes = [P, P, I64, I64, I64, P]
        lib.oracle_linear_logits.restype = None
        lib.oracle_linear_grads.argtypes = [P, P, P, I64, I64, I64, P, P]
        lib.oracle_linear_grads.restype = None
        lib.oracle_entropy.argtypes = [P, I64, I64, P, P]
        lib.oracle_entropy.restype = None
        _lib = lib
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def ce_forward(z, target, eps: float = 0.0, ignore_idx: int = -100):
    """Per-row loss, m, lse, bad flags and N_v of float64 logits z [n, V]."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    n, v = z.shape
    y = np.ascontiguousarray(target, dtype=np.int64)
    loss, m, lse = np.empty(n), np.empty(n), np.empty(n)
    bad = np.empty(n, dtype=np.int32)
    nv = _load().oracle_ce_forward(_p(z), n, v, v, _p(y), float(eps), int(ignore_idx), _p(loss), _p(m),
                                   _p(lse), _p(bad))
    return dict(loss_rows=loss, m=m, lse=lse, bad=bad.astype(bool), n_valid=int(nv))


def ce_backward(z, target, lse, g_rows, eps: float = 0.0, ignore_idx: int = -100):
    z = np.ascontiguousarray(z, dtype=np.float64)
    n, v = z.shape
    y = np.ascontiguousarray(target, dtype=np.int64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    g = np.ascontiguousarray(g_rows, dtype=np.float64)
    dz = np.empty((n, v))
    _load().oracle_ce_backward(_p(z), n, v, v, _p(y), _p(lse), _p(g), float(eps), int(ignore_idx), _p(dz))
    return dz


def linear_logits(x, w):
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    n, h = x.shape
    v = w.shape[0]
    z = np.empty((n, v))
    _load().oracle_linear_logits(_p(x), _p(w), n, h, v, _p(z))
    return z


def linear_grads(dz, x, w):
    """dX = dZ W and dW = dZ^T X in float64."""
    dz = np.ascontiguousarray(dz, dtype=np.float64)
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    n, h = x.shape
    v = w.shape[0]
    dx, dw = np.empty((n, h)), np.empty((v, h))
    _load().oracle_linear_grads(_p(dz), _p(x), _p(w), n, h, v, _p(dx), _p(dw))
    return dx, dw


def entropy(z, lse):
    z = np.ascontiguousarray(z, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    n, v = z.shape
    ent = np.empty(n)
    _load().oracle_entropy(_p(z), n, v, _p(lse), _p(ent))
    return ent

"""fp64 CPU oracle for row-wise RMSNorm / LayerNorm, forward and backward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path never
imports this package, and this package imports nothing from the product.

The arithmetic lives in ``norm_oracle.c`` (plain C, fp64, one row at a time,
exactly the definitions on the "SOTA normalization performance with
torch.compile" page, section "How Did Torch.compile Catch Quack?", and the
"Fused RMSNorm" page, section "What it is").  This module only compiles that
file with gcc and marshals arrays through ctypes.

Inputs are promoted to float64 from values already rounded to the storage
dtype (the promotion is exact); outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "norm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile norm_oracle.c into liboracle.so (OpenMP if gcc supports it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            inp = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
            i64, d = ctypes.c_int64, ctypes.c_double
            f64p = ctypes.c_void_p  # may be NULL
            lib.oracle_rmsnorm_fwd.argtypes = [inp, inp, i64, i64, d, f64p, f64p]
            lib.oracle_layernorm_fwd.argtypes = [inp, inp, inp, i64, i64, d, f64p, f64p, f64p]
            lib.oracle_rmsnorm_bwd.argtypes = [inp, inp, inp, i64, i64, d, f64p, f64p]
            lib.oracle_layernorm_bwd.argtypes = [inp, inp, inp, i64, i64, d, f64p, f64p, f64p]
            lib.oracle_rmsnorm_fwd.restype = None
            lib.oracle_layernorm_fwd.restype = None
            lib.oracle_rmsnorm_bwd.restype = ctypes.c_int
            lib.oracle_layernorm_bwd.restype = ctypes.c_int
            lib.oracle_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch tensor: exact promotion of its dtype to float64
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data


def threads() -> int:
    """Host threads the oracle runs on."""
    return _load().oracle_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def rmsnorm_fwd(x, gamma, eps: float):
    """Returns (y [M,N] f64, rstd [M] f64)."""
    x, gamma = _f64(x), _f64(gamma)
    M, N = x.shape
    y = np.empty((M, N), np.float64)
    rstd = np.empty(M, np.float64)
    _load().oracle_rmsnorm_fwd(x, gamma, M, N, eps, _ptr(y), _ptr(rstd))
    return y, rstd


def layernorm_fwd(x, gamma, beta, eps: float):
    """Returns (y [M,N] f64, mean [M] f64, rstd [M] f64)."""
    x, gamma, beta = _f64(x), _f64(gamma), _f64(beta)
    M, N = x.shape
    y = np.empty((M, N), np.float64)
    mean = np.empty(M, np.float64)
    rstd = np.empty(M, np.float64)
    _load().oracle_layernorm_fwd(x, gamma, beta, M, N, eps, _ptr(y), _ptr(mean), _ptr(rstd))
    return y, mean, rstd


def rmsnorm_bwd(dy, x, gamma, eps: float, want_dx: bool = True, want_dgamma: bool = True, dres=None):
    """Returns (dx [M,N] f64 or None, dgamma [N] f64 or None).  dres: the
    gradient reaching the normalised rows from a residual stream (see
    residual_add), added to dx."""
    dy, x, gamma = _f64(dy), _f64(x), _f64(gamma)
    M, N = x.shape
    dx = np.empty((M, N), np.float64) if want_dx else None
    dg = np.empty(N, np.float64) if want_dgamma else None
    if _load().oracle_rmsnorm_bwd(dy, x, gamma, M, N, eps, _ptr(dx), _ptr(dg)) != 0:
        raise MemoryError("oracle: out of host memory")
    if dx is not None and dres is not None:
        dx += _f64(dres)
    return dx, dg


def layernorm_bwd(dy, x, gamma, eps: float, want_dx: bool = True, want_dparams: bool = True, dres=None):
    """Returns (dx [M,N] f64 or None, dgamma [N] f64 or None, dbeta [N] f64 or
    None).  dres as for rmsnorm_bwd."""
    dy, x, gamma = _f64(dy), _f64(x), _f64(gamma)
    M, N = x.shape
    dx = np.empty((M, N), np.float64) if want_dx else None
    dg = np.empty(N, np.float64) if want_dparams else None
    db = np.empty(N, np.float64) if want_dparams else None
    if _load().oracle_layernorm_bwd(dy, x, gamma, M, N, eps, _ptr(dx), _ptr(dg), _ptr(db)) != 0:
        raise MemoryError("oracle: out of host memory")
    if dx is not None and dres is not None:
        dx += _f64(dres)
    return dx, dg, db


def residual_add(x, r, dtype=None):
    """The residual sum a fused "add + norm" normalises and stores: h = x + r,
    rounded once (round to nearest even) to `dtype`, the storage type of x and
    r ("bf16", "fp16", "fp32"; None keeps the exact fp64 sum, for
    finite-difference checks).  The norm is then taken of the stored h -- the
    result an unfused h = x + r followed by the norm gives.

    x + r is formed in fp64; for two values of one of these types the fp64 sum
    is either exact, or (exponents more than 29 apart for fp32, 45 for bf16)
    so far from a rounding midpoint of the type that rounding it once more
    gives the same value as rounding the exact sum.  Returns a CPU torch tensor
    of `dtype` (or an fp64 numpy array)."""
    s = _f64(x) + _f64(r)
    if dtype is None:
        return s
    import torch
    t = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[dtype]
    return torch.from_numpy(s).to(t)

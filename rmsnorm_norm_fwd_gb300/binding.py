"""Thin Python binding over libgbnorm.so (include/gbnorm.h).

Argument marshalling only: tensors are checked (CUDA, contiguous, matching
dtype and shape), outputs and the backward workspace are allocated with torch's
caching allocator when the caller does not pass them, and the call goes to the
C ABI on torch's current stream.  Every step of the computation runs in the
library's CUDA kernels; there is no other implementation to fall back to, and
importing this module fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("GBNORM_LIB", os.path.join(_HERE, "libgbnorm.so"))

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libgbnorm.so not found at {LIB_PATH}: build it first "
        "(python -m rmsnorm_norm_fwd_gb300.build, or __graft_entry__.build()).")

lib = ctypes.CDLL(LIB_PATH)

_vp, _i64, _int, _f, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
lib.rmsnorm_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _int, _f, _vp]
lib.layernorm_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _f, _vp]
lib.norm_bwd_workspace_size.argtypes = [_int, _i64, _i64, _int]
lib.norm_bwd_workspace_size.restype = _sz
lib.rmsnorm_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _int, _vp]
lib.layernorm_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _int, _vp]
lib.norm_fwd_ex.argtypes = [_int, _i64, _i64, _f, _vp, _i64, _int, _vp, _i64, _vp, _i64, _vp, _vp, _int,
                            _vp, _i64, _int, _vp, _vp, _vp]
lib.norm_bwd_ex_workspace_size.argtypes = [_int, _i64, _i64]
lib.norm_bwd_ex_workspace_size.restype = _sz
lib.norm_bwd_ex.argtypes = [_int, _i64, _i64, _vp, _i64, _int, _vp, _i64, _int, _vp, _i64, _vp, _int, _vp, _vp,
                            _vp, _i64, _vp, _vp, _vp, _sz, _vp]
lib.gbnorm_status_string.argtypes = [_int]
lib.gbnorm_status_string.restype = ctypes.c_char_p
lib.gbnorm_variant_name.argtypes = [_int, _int, _i64, _i64, _int, _int, ctypes.c_char_p, _sz]
lib.gbnorm_force_variant.argtypes = [_int, _int, _int, ctypes.c_char_p]
lib.gbnorm_variant_count.argtypes = [_int, _int, _int]
lib.gbnorm_variant_at.argtypes = [_int, _int, _int, _int]
lib.gbnorm_variant_at.restype = ctypes.c_char_p
lib.gbnorm_read_fault.argtypes = [_int, ctypes.POINTER(ctypes.c_int)]
lib.gbnorm_set_grid_limit.argtypes = [_int]
lib.gbnorm_ex_variant_count.argtypes = [_int, _int]
lib.gbnorm_ex_variant_at.argtypes = [_int, _int, _int]
lib.gbnorm_ex_variant_at.restype = ctypes.c_char_p
lib.gbnorm_ex_force_variant.argtypes = [_int, _int, ctypes.c_char_p]
lib.gbnorm_ex_last_variant.argtypes = [_int, ctypes.c_char_p, _sz]
for _fn in ("rmsnorm_fwd", "layernorm_fwd", "rmsnorm_bwd", "layernorm_bwd", "norm_fwd_ex", "norm_bwd_ex",
            "gbnorm_variant_name",
            "gbnorm_force_variant", "gbnorm_variant_count", "gbnorm_read_fault",
            "gbnorm_set_grid_limit", "gbnorm_ex_variant_count", "gbnorm_ex_force_variant",
            "gbnorm_ex_last_variant"):
    getattr(lib, _fn).restype = _int

GBNORM_OK = 0
DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
DTYPE_NAME = {"fp32": 0, "fp16": 1, "bf16": 2}


class GbnormError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {lib.gbnorm_status_string(status).decode()} (status {status})")
        self.status = status


def _check(fn: str, status: int) -> None:
    if status != GBNORM_OK:
        raise GbnormError(fn, status)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _mat(name, t, dtype=None):
    if not (t.is_cuda and t.dim() == 2 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous 2-D CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}")
    return t


def _vec(name, t, n, dtype):
    if not (t.is_cuda and t.dim() == 1 and t.is_contiguous() and t.numel() == n and t.dtype == dtype):
        raise ValueError(f"{name} must be a contiguous 1-D CUDA {dtype} tensor of {n} elements")
    return t


def _opt_vec(name, t, n, dtype):
    return None if t is None else _vec(name, t, n, dtype)


def rmsnorm_fwd(x, gamma, eps: float, y=None, rstd=None, save_stats: bool = True, stream=None):
    """y = x * rstd * gamma per row (gamma None: 1); returns (y, rstd) (rstd None if not saved)."""
    _mat("x", x)
    M, N = x.shape
    _opt_vec("gamma", gamma, N, x.dtype)
    y = torch.empty_like(x) if y is None else _mat("y", y, x.dtype)
    if rstd is None and save_stats:
        rstd = torch.empty(M, device=x.device, dtype=torch.float32)
    _check("rmsnorm_fwd", lib.rmsnorm_fwd(_ptr(x), _ptr(gamma), _ptr(y), _ptr(rstd), M, N,
                                          DTYPE_CODE[x.dtype], float(eps), _stream(stream)))
    return y, rstd


def layernorm_fwd(x, gamma, beta, eps: float, y=None, mean=None, rstd=None, save_stats: bool = True,
                  stream=None):
    """y = (x - mean) * rstd * gamma + beta per row (gamma None: 1, beta None: 0);
    returns (y, mean, rstd)."""
    _mat("x", x)
    M, N = x.shape
    _opt_vec("gamma", gamma, N, x.dtype)
    _opt_vec("beta", beta, N, x.dtype)
    y = torch.empty_like(x) if y is None else _mat("y", y, x.dtype)
    if save_stats:
        mean = torch.empty(M, device=x.device, dtype=torch.float32) if mean is None else mean
        rstd = torch.empty(M, device=x.device, dtype=torch.float32) if rstd is None else rstd
    _check("layernorm_fwd", lib.layernorm_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(mean),
                                              _ptr(rstd), M, N, DTYPE_CODE[x.dtype], float(eps),
                                              _stream(stream)))
    return y, mean, rstd


def norm_bwd_workspace_size(is_layernorm: bool, M: int, N: int, dtype) -> int:
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else DTYPE_NAME.get(dtype, dtype)
    return int(lib.norm_bwd_workspace_size(int(bool(is_layernorm)), M, N, code))


def _workspace(is_ln, x, workspace):
    M, N = x.shape
    need = norm_bwd_workspace_size(is_ln, M, N, x.dtype)
    if need == 0:
        raise GbnormError("norm_bwd_workspace_size", 2)
    if workspace is None:
        workspace = torch.empty(need, device=x.device, dtype=torch.uint8)
    return workspace, workspace.numel() * workspace.element_size()


def rmsnorm_bwd(dy, x, gamma, rstd, dx=None, dgamma=None, workspace=None, stream=None,
                need_dgamma: bool = True):
    """Returns (dx, dgamma) with dgamma in float32 (gamma None: 1; need_dgamma
    False with no dgamma given: not produced, None)."""
    _mat("x", x)
    M, N = x.shape
    _mat("dy", dy, x.dtype)
    _opt_vec("gamma", gamma, N, x.dtype)
    _vec("rstd", rstd, M, torch.float32)
    dx = torch.empty_like(x) if dx is None else _mat("dx", dx, x.dtype)
    if dgamma is None and need_dgamma:
        dgamma = torch.empty(N, device=x.device, dtype=torch.float32)
    ws, wsb = _workspace(False, x, workspace)
    _check("rmsnorm_bwd", lib.rmsnorm_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(rstd), _ptr(dx),
                                          _ptr(dgamma), _ptr(ws), wsb, M, N, DTYPE_CODE[x.dtype],
                                          _stream(stream)))
    return dx, dgamma


def layernorm_bwd(dy, x, gamma, mean, rstd, dx=None, dgamma=None, dbeta=None, workspace=None,
                  stream=None, need_dgamma: bool = True, need_dbeta: bool = True):
    """Returns (dx, dgamma, dbeta) with dgamma and dbeta in float32 (gamma None:
    1; a sum not needed and not given is not produced, None)."""
    _mat("x", x)
    M, N = x.shape
    _mat("dy", dy, x.dtype)
    _opt_vec("gamma", gamma, N, x.dtype)
    _vec("mean", mean, M, torch.float32)
    _vec("rstd", rstd, M, torch.float32)
    dx = torch.empty_like(x) if dx is None else _mat("dx", dx, x.dtype)
    if dgamma is None and need_dgamma:
        dgamma = torch.empty(N, device=x.device, dtype=torch.float32)
    if dbeta is None and need_dbeta:
        dbeta = torch.empty(N, device=x.device, dtype=torch.float32)
    ws, wsb = _workspace(True, x, workspace)
    _check("layernorm_bwd", lib.layernorm_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(mean), _ptr(rstd),
                                              _ptr(dx), _ptr(dgamma), _ptr(dbeta), _ptr(ws), wsb, M, N,
                                              DTYPE_CODE[x.dtype], _stream(stream)))
    return dx, dgamma, dbeta


# ---------------------------------------------------------------------------- general form
def _rows(name, t):
    """A 2-D CUDA tensor whose rows are contiguous (any row stride): (ptr, ld)."""
    if not (t.is_cuda and t.dim() == 2 and (t.stride(1) == 1 or t.shape[1] <= 1)):
        raise ValueError(f"{name} must be a 2-D CUDA tensor with unit column stride")
    return t.data_ptr(), max(t.stride(0), t.shape[1])


def _code(t, default):
    return DTYPE_CODE[t.dtype] if t is not None else DTYPE_CODE[default]


def norm_fwd_ex(is_layernorm: bool, x, gamma, beta, eps: float, residual=None, store_h: bool = True,
                y_dtype=None, y=None, h=None, mean=None, rstd=None, save_stats: bool = True, stream=None):
    """General forward: rows of x (any row stride), optional residual rows
    (x's dtype) added first, gamma / beta of their own dtype, y of y_dtype
    (default x's).  Returns (y, h, mean, rstd); h (the stored residual sum) is
    None without a residual or with store_h False, mean None for RMSNorm."""
    px, ldx = _rows("x", x)
    M, N = x.shape
    pr, ldr = _rows("residual", residual) if residual is not None else (None, N)
    if residual is not None and (residual.dtype != x.dtype or residual.shape != x.shape):
        raise ValueError("residual must match x in shape and dtype")
    if gamma is not None and beta is not None and gamma.dtype != beta.dtype:
        raise ValueError("gamma and beta must share a dtype")
    pdt = gamma.dtype if gamma is not None else (beta.dtype if beta is not None else x.dtype)
    for nm, v in (("gamma", gamma), ("beta", beta)):
        if v is not None:
            _vec(nm, v, N, pdt)
    if y is None:
        y = torch.empty(M, N, device=x.device, dtype=y_dtype or x.dtype)
    py, ldy = _rows("y", y)
    if residual is not None and store_h and h is None:
        h = torch.empty_like(x, memory_format=torch.contiguous_format)
    ph, ldh = _rows("h", h) if h is not None else (None, N)
    if save_stats:
        rstd = torch.empty(M, device=x.device, dtype=torch.float32) if rstd is None else rstd
        if is_layernorm:
            mean = torch.empty(M, device=x.device, dtype=torch.float32) if mean is None else mean
    _check("norm_fwd_ex", lib.norm_fwd_ex(int(bool(is_layernorm)), M, N, float(eps), px, ldx, DTYPE_CODE[x.dtype],
                                          pr, ldr, ph, ldh, _ptr(gamma), _ptr(beta), DTYPE_CODE[pdt], py, ldy,
                                          DTYPE_CODE[y.dtype], _ptr(mean), _ptr(rstd), _stream(stream)))
    return y, h, mean, rstd


def norm_bwd_ex_workspace_size(is_layernorm: bool, M: int, N: int) -> int:
    return int(lib.norm_bwd_ex_workspace_size(int(bool(is_layernorm)), M, N))


def norm_bwd_ex(is_layernorm: bool, dy, x, gamma, mean, rstd, dres=None, dx=None, dgamma=None, dbeta=None,
                workspace=None, need_dgamma: bool = True, need_dbeta: bool = True, stream=None):
    """General backward: dy (y's dtype) and x (the normalised rows, h after a
    residual add) with any row strides, gamma of its own dtype, dres (x's
    dtype) added into dx.  Returns (dx, dgamma, dbeta) with dx of x's dtype."""
    pdy, lddy = _rows("dy", dy)
    px, ldx = _rows("x", x)
    M, N = x.shape
    if dy.shape != x.shape:
        raise ValueError("dy must match x in shape")
    pdr, lddr = _rows("dres", dres) if dres is not None else (None, N)
    if dres is not None and (dres.dtype != x.dtype or dres.shape != x.shape):
        raise ValueError("dres must match x in shape and dtype")
    if gamma is not None:
        _vec("gamma", gamma, N, gamma.dtype)
    _vec("rstd", rstd, M, torch.float32)
    if is_layernorm:
        _vec("mean", mean, M, torch.float32)
    if dx is None:
        dx = torch.empty(M, N, device=x.device, dtype=x.dtype)
    pdx, lddx = _rows("dx", dx)
    if dgamma is None and need_dgamma:
        dgamma = torch.empty(N, device=x.device, dtype=torch.float32)
    if is_layernorm and dbeta is None and need_dbeta:
        dbeta = torch.empty(N, device=x.device, dtype=torch.float32)
    need = norm_bwd_ex_workspace_size(is_layernorm, M, N)
    if need == 0:
        raise GbnormError("norm_bwd_ex_workspace_size", 2)
    if workspace is None:
        workspace = torch.empty(need, device=x.device, dtype=torch.uint8)
    _check("norm_bwd_ex", lib.norm_bwd_ex(int(bool(is_layernorm)), M, N, pdy, lddy, DTYPE_CODE[dy.dtype], px, ldx,
                                          DTYPE_CODE[x.dtype], pdr, lddr, _ptr(gamma), _code(gamma, x.dtype),
                                          _ptr(mean if is_layernorm else None), _ptr(rstd), pdx, lddx,
                                          _ptr(dgamma), _ptr(dbeta if is_layernorm else None), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream)))
    return dx, dgamma, (dbeta if is_layernorm else None)


def variant_name(is_layernorm: bool, direction: int, M: int, N: int, dtype, aligned: bool = True) -> str:
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else DTYPE_NAME.get(dtype, dtype)
    buf = ctypes.create_string_buffer(64)
    _check("gbnorm_variant_name", lib.gbnorm_variant_name(int(bool(is_layernorm)), direction, M, N,
                                                          code, int(aligned), buf, 64))
    return buf.value.decode()


def force_variant(is_layernorm: bool, direction: int, dtype, name: str | None) -> None:
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else DTYPE_NAME.get(dtype, dtype)
    _check("gbnorm_force_variant", lib.gbnorm_force_variant(
        int(bool(is_layernorm)), direction, code, None if not name else name.encode()))


def variants(is_layernorm: bool, direction: int, dtype) -> list[str]:
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else DTYPE_NAME.get(dtype, dtype)
    n = lib.gbnorm_variant_count(int(bool(is_layernorm)), direction, code)
    return [lib.gbnorm_variant_at(int(bool(is_layernorm)), direction, code, i).decode() for i in range(n)]


def ex_variants(is_layernorm: bool, direction: int) -> list[str]:
    """Names of the general form's kernels for (op, direction); the last is "exe"."""
    n = lib.gbnorm_ex_variant_count(int(bool(is_layernorm)), direction)
    return [lib.gbnorm_ex_variant_at(int(bool(is_layernorm)), direction, i).decode() for i in range(n)]


def ex_force_variant(is_layernorm: bool, direction: int, name: str | None) -> None:
    """Make later general-form calls launch `name` where it can serve them (None: no override)."""
    _check("gbnorm_ex_force_variant", lib.gbnorm_ex_force_variant(
        int(bool(is_layernorm)), direction, None if not name else name.encode()))


def ex_last_variant(direction: int) -> str:
    """The kernel this thread's last norm_fwd_ex (0) / norm_bwd_ex (1) launched ("" for none)."""
    buf = ctypes.create_string_buffer(64)
    _check("gbnorm_ex_last_variant", lib.gbnorm_ex_last_variant(direction, buf, 64))
    return buf.value.decode()


def read_fault(reset: bool = True) -> int:
    """The device fault word (nonzero if a kernel's bounded wait gave up)."""
    v = ctypes.c_int(0)
    _check("gbnorm_read_fault", lib.gbnorm_read_fault(int(reset), ctypes.byref(v)))
    return v.value


def set_grid_limit(max_ctas: int) -> None:
    """Cap the persistent grid of later launches (0 removes the cap); tests/tuning."""
    _check("gbnorm_set_grid_limit", lib.gbnorm_set_grid_limit(int(max_ctas)))

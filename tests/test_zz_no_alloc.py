"""rmsnorm_bwd_noalloc: the RMSNorm backward for callers that cannot allocate
device memory (an allocator callback, a plugin under a fixed memory budget, a
hot path where cudaMalloc is not allowed).  It keeps its dgamma partial rows
in a fixed scratch array inside the library instead of a caller workspace.

It runs the same kernels with the same number of partial rows as
rmsnorm_bwd, so the two must agree bitwise; dgamma is also held to the fp64
oracle's column sums (1e-3 relative L2).  The calls run in an order that
would expose stale scratch: a shape with few partial rows first, then one
with more, then one without gamma and without dgamma.  This file is collected
last so that a run stopping at the first failure has already run every other
test (GPU)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from rmsnorm_norm_fwd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

GBNORM_ERR_WORKSPACE = 3
SCRATCH_BYTES = 16 << 20


def _lib():
    from rmsnorm_norm_fwd_gb300 import binding
    lib = binding.lib
    vp, i64, i = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.rmsnorm_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i, vp]
    lib.rmsnorm_bwd_noalloc.restype = i
    return binding, lib


def _ptr(t):
    return None if t is None else t.data_ptr()


def test_noalloc_matches_workspace_entry_point():
    binding, lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    # (M, N, dtype, with gamma): few partial rows, then more, then no gamma/dgamma.
    cases = ((200, 2048, "bf16", True), (9001, 2048, "bf16", True), (777, 5120, "fp16", True),
             (4099, 1024, "bf16", False))
    for (M, N, dtype, with_gamma) in cases:
        inp = make_inputs(M, N, dtype=dtype, op="rms")
        x, dy = inp.x.cuda(), inp.dy.cuda()
        gam = inp.gamma.cuda() if with_gamma else None
        _, rstd = binding.rmsnorm_fwd(x, gam, inp.eps)
        dx_ref, dg_ref = binding.rmsnorm_bwd(dy, x, gam, rstd, need_dgamma=with_gamma)
        dx = torch.full_like(x, float("nan"))
        dg = torch.full((N,), float("nan"), device="cuda") if with_gamma else None
        st = lib.rmsnorm_bwd_noalloc(_ptr(dy), _ptr(x), _ptr(gam), _ptr(rstd), _ptr(dx), _ptr(dg),
                                     M, N, binding.DTYPE_CODE[x.dtype], stream)
        assert st == 0, lib.gbnorm_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(dx, dx_ref), (M, N, dtype)
        if with_gamma:
            assert torch.equal(dg, dg_ref), (M, N, dtype)
            _, dg_or = oracle.rmsnorm_bwd(inp.dy, inp.x, inp.gamma, inp.eps, want_dx=False)
            got = dg.double().cpu().numpy()
            assert np.linalg.norm(got - dg_or) <= 1e-3 * np.linalg.norm(dg_or), (M, N, dtype)
    assert binding.read_fault(reset=True) == 0


def test_noalloc_refuses_shapes_beyond_its_scratch():
    binding, lib = _lib()
    M, N = 200, 65536  # element-wise path worst case: 152 partial rows of 256 KiB
    need = binding.norm_bwd_workspace_size(False, M, N, torch.bfloat16)
    assert need > SCRATCH_BYTES
    x = torch.zeros(M, N, device="cuda", dtype=torch.bfloat16)
    gam = torch.ones(N, device="cuda", dtype=torch.bfloat16)
    rstd = torch.ones(M, device="cuda")
    dx = torch.empty_like(x)
    dg = torch.empty(N, device="cuda")
    st = lib.rmsnorm_bwd_noalloc(x.data_ptr(), x.data_ptr(), gam.data_ptr(), rstd.data_ptr(),
                                 dx.data_ptr(), dg.data_ptr(), M, N, 2,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == GBNORM_ERR_WORKSPACE

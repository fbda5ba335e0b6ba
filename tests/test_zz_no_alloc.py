"""rmsnorm_bwd_noalloc: the RMSNorm backward for callers that cannot allocate
device memory (an allocator callback, a plugin under a fixed memory budget, a
hot path where cudaMalloc is not allowed).  It keeps its dgamma partial rows
in a fixed scratch array inside the library instead of a caller workspace.

Called through the C ABI and checked against rmsnorm_bwd (the workspace entry
point) on two calls in a row, with the parity tests' tolerances: dx within 2
units in the last place of the output dtype, dgamma within 1e-3 of the L2
norm.  This file is collected last so that a run stopping at the first
failure has already run every other test (GPU)."""
import ctypes

import pytest
import torch

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


def _ulp(t):
    """Spacing of t's dtype at |t| (float64 tensor)."""
    info = torch.finfo(t.dtype)
    a = t.double().abs().clamp_min(info.tiny)
    return torch.exp2(torch.floor(torch.log2(a)) - {torch.bfloat16: 7, torch.float16: 10,
                                                     torch.float32: 23}[t.dtype])


def test_noalloc_matches_workspace_entry_point():
    binding, lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    # Two calls in a row, different shapes and dtypes.
    for (M, N, dtype) in ((4099, 2048, "bf16"), (777, 5120, "fp16")):
        inp = make_inputs(M, N, dtype=dtype, op="rms")
        x, dy, gam = inp.x.cuda(), inp.dy.cuda(), inp.gamma.cuda()
        _, rstd = binding.rmsnorm_fwd(x, gam, inp.eps)
        dx_ref, dg_ref = binding.rmsnorm_bwd(dy, x, gam, rstd)
        dx = torch.empty_like(x)
        dg = torch.full((N,), float("nan"), device="cuda")
        st = lib.rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), gam.data_ptr(), rstd.data_ptr(),
                                     dx.data_ptr(), dg.data_ptr(), M, N,
                                     binding.DTYPE_CODE[x.dtype], stream)
        assert st == 0, lib.gbnorm_status_string(st)
        torch.cuda.synchronize()
        err = (dx.double() - dx_ref.double()).abs()
        assert torch.all(err <= 2 * _ulp(dx_ref)), float(err.max())
        rel = torch.linalg.norm(dg.double() - dg_ref.double()) / torch.linalg.norm(dg_ref.double())
        assert rel <= 1e-3, float(rel)
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

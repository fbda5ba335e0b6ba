"""The general form (norm_fwd_ex / norm_bwd_ex through the C ABI) against the
fp64 oracle: a storage type per tensor (rows, parameters, output), rows with
their own strides, and the fused residual add, forward and backward, on the
vector path and the element-wise path (GPU)."""
import re

import numpy as np
import pytest
import torch

import oracle
from parity_util import compare
from rmsnorm_norm_fwd_gb300.inputs import DTYPES, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_fault():
    import rmsnorm_norm_fwd_gb300 as g
    g.read_fault(reset=True)
    yield
    assert g.read_fault(reset=True) == 0


def _strided(t, pad):
    """t on the GPU as a view with row stride N + pad (the padding holds NaN)."""
    M, N = t.shape
    buf = torch.full((M, N + pad), float("nan"), dtype=t.dtype, device="cuda")
    v = buf[:, :N]
    v.copy_(t.to("cuda"))
    return v


def _vec(*ts):
    return all(t is None or (t.data_ptr() % 16 == 0 and (t.stride(0) * t.element_size()) % 16 == 0)
               for t in ts)


def run_ex(op, inp, pad=0, y_dtype=None, residual=None, dres=None, store_h=True, check_path=True):
    """Forward and backward through the general form; returns (host outputs,
    variants).  With a residual, inp.x is x and the backward differentiates at
    the stored h; without one, x itself."""
    import rmsnorm_norm_fwd_gb300 as g
    ln = op == "ln"
    x = _strided(inp.x, pad)
    r = _strided(residual, pad) if residual is not None else None
    gam, bet = inp.gamma.cuda(), inp.beta.cuda() if ln else None
    y = _strided(torch.empty(inp.x.shape, dtype=DTYPES[y_dtype or inp.dtype]), pad + 8)
    y, h, mean, rstd = g.norm_fwd_ex(ln, x, gam, bet, inp.eps, residual=r, store_h=store_h, y=y)
    vf = g.ex_last_variant(0)
    dy = _strided(inp.dy, pad)
    xb = h if h is not None else x
    if residual is not None and h is None:  # h not stored: the oracle's, for the backward
        xb = _strided(oracle.residual_add(inp.x, residual, inp.dtype), pad)
    dr = _strided(dres, pad) if dres is not None else None
    dx = _strided(torch.empty(inp.x.shape, dtype=inp.x.dtype), pad + 16)
    dx, dg, db = g.norm_bwd_ex(ln, dy, xb, gam, mean, rstd, dres=dr, dx=dx)
    vb = g.ex_last_variant(1)
    torch.cuda.synchronize()
    out = {"y": y.cpu(), "rstd": rstd.cpu(), "dx": dx.cpu(), "dgamma": dg.cpu()}
    if ln:
        out.update(mean=mean.cpu(), dbeta=db.cpu())
    if h is not None:
        out["h"] = h.cpu()
    assert vf and vb
    # the vector kernels hold rows of up to 16384 elements
    N = inp.x.shape[1]
    vec_f = _vec(x, r, h, y) and gam.data_ptr() % 16 == 0 and N % 8 == 0 and N <= 16384
    vec_b = _vec(dy, xb, dr, dx) and N % 8 == 0 and N <= 16384
    assert not check_path or ((vf != "exe") == vec_f and (vb != "exe") == vec_b), (vf, vb)
    return out, (vf, vb)


MIXED = [("bf16", "fp32", "bf16"), ("fp16", "fp32", "fp16"), ("fp32", "fp32", "bf16"),
         ("bf16", "bf16", "fp32"), ("fp32", "bf16", "fp16")]


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("types", MIXED, ids=["-".join(t) for t in MIXED])
@pytest.mark.parametrize("N", [1000, 4096, 5120, 16384, 32768])
def test_mixed_dtypes(op, types, N):
    """Rows, parameters and output each in their own type (x / gamma / y):
    y is held to its own type's tolerance, dx to x's."""
    xdt, pdt, ydt = types
    M = 301 if N <= 8192 else 37
    inp = make_inputs(M, N, dtype=xdt, dist="llm" if N >= 4096 else op, op=op, param_dtype=pdt, dy_dtype=ydt)
    out, variants = run_ex(op, inp, y_dtype=ydt)
    compare(op, inp, out, variants=variants, y_dtype=ydt).assert_ok()


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N,pad", [(384, 8), (384, 3), (4096, 64), (4096, 1), (65536, 8)])
def test_strided_rows(op, dtype, N, pad):
    """Rows inside wider buffers (x, y, dy and dx each with its own stride);
    a padding that breaks 16-byte rows takes the element-wise kernels."""
    M = 129 if N <= 4096 else 9
    inp = make_inputs(M, N, dtype=dtype, dist="llm" if N >= 4096 else op, op=op)
    out, variants = run_ex(op, inp, pad=pad)
    compare(op, inp, out, variants=variants).assert_ok()


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("N", [1000, 2048, 8192])
@pytest.mark.parametrize("store_h", [True, False])
def test_residual_add(op, dtype, N, store_h):
    """h = x + r rounded once to the storage type, stored (bit-identical to the
    oracle's), normalised; backward at h with the residual stream's gradient
    added into dx."""
    M = 211
    inp = make_inputs(M, N, dtype=dtype, dist=op, op=op)
    res = make_inputs(M, N, dtype=dtype, dist="rms", op=op, seed=99).x
    dres = make_inputs(M, N, dtype=dtype, dist="rms", op=op, seed=98).dy
    out, variants = run_ex(op, inp, residual=res, dres=dres, store_h=store_h)
    h_ref = oracle.residual_add(inp.x, res, dtype)
    if store_h:
        assert torch.equal(out["h"], h_ref)
    inp_h = make_inputs(M, N, dtype=dtype, dist=op, op=op)
    inp_h.x = h_ref
    compare(op, inp_h, out, variants=variants, dres=dres).assert_ok()


@pytest.mark.parametrize("op", ["rms", "ln"])
def test_residual_in_place(op):
    """h written over r and dx over dres (the usual layout of a residual
    stream): the same results as with separate buffers."""
    import rmsnorm_norm_fwd_gb300 as g
    ln = op == "ln"
    M, N = 333, 4096
    inp = make_inputs(M, N, dtype="bf16", op=op, dist=op)
    x, gam = inp.x.cuda(), inp.gamma.cuda()
    bet = inp.beta.cuda() if ln else None
    r = make_inputs(M, N, dtype="bf16", seed=7).x.cuda()
    dres = make_inputs(M, N, dtype="bf16", seed=8).dy.cuda()
    dy = inp.dy.cuda()
    y1, h1, m1, r1 = g.norm_fwd_ex(ln, x, gam, bet, inp.eps, residual=r)
    dx1, dg1, db1 = g.norm_bwd_ex(ln, dy, h1, gam, m1, r1, dres=dres)
    r2, dres2 = r.clone(), dres.clone()
    y2, h2, m2, s2 = g.norm_fwd_ex(ln, x, gam, bet, inp.eps, residual=r2, h=r2)
    assert h2.data_ptr() == r2.data_ptr()
    dx2, dg2, db2 = g.norm_bwd_ex(ln, dy, h2, gam, m2, s2, dres=dres2, dx=dres2)
    torch.cuda.synchronize()
    assert torch.equal(h1, r2) and torch.equal(y1, y2) and torch.equal(dx1, dres2)
    assert torch.equal(dg1, dg2) and (not ln or torch.equal(db1, db2))


@pytest.mark.parametrize("op", ["rms", "ln"])
def test_optional_parameters_and_empty(op):
    """NULL gamma / beta are 1 / 0; M = 0 launches nothing and gives zero
    parameter gradients."""
    import rmsnorm_norm_fwd_gb300 as g
    ln = op == "ln"
    M, N = 64, 2048
    inp = make_inputs(M, N, dtype="bf16", op=op, dist=op)
    inp.gamma = torch.ones_like(inp.gamma)
    inp.beta = torch.zeros_like(inp.beta)
    x, dy = inp.x.cuda(), inp.dy.cuda()
    y, _, mean, rstd = g.norm_fwd_ex(ln, x, None, None, inp.eps)
    vf = g.ex_last_variant(0)
    dx, dg, db = g.norm_bwd_ex(ln, dy, x, None, mean, rstd)
    vb = g.ex_last_variant(1)
    torch.cuda.synchronize()
    out = {"y": y.cpu(), "rstd": rstd.cpu(), "dx": dx.cpu(), "dgamma": dg.cpu()}
    if ln:
        out.update(mean=mean.cpu(), dbeta=db.cpu())
    assert vf.startswith("exrf") and vb.startswith("exrb"), (vf, vb)
    compare(op, inp, out, variants=(vf, vb)).assert_ok()
    e = torch.empty(0, N, device="cuda", dtype=torch.bfloat16)
    dge = torch.full((N,), 5.0, device="cuda")
    _, _, me, re_ = g.norm_fwd_ex(ln, e, None, None, inp.eps)
    assert g.ex_last_variant(0) == ""
    g.norm_bwd_ex(ln, e, e, None, me, re_, dgamma=dge)
    assert g.ex_last_variant(1) == ""
    torch.cuda.synchronize()
    assert torch.all(dge == 0)


def test_ex_deterministic():
    import rmsnorm_norm_fwd_gb300 as g
    inp = make_inputs(1000, 5120, dtype="bf16", op="ln", dist="llm", param_dtype="fp32")
    x, gam, bet, dy = inp.x.cuda(), inp.gamma.cuda(), inp.beta.cuda(), inp.dy.cuda()
    outs = []
    for _ in range(2):
        y, _, m, r = g.norm_fwd_ex(True, x, gam, bet, inp.eps)
        outs.append((y, m, r) + g.norm_bwd_ex(True, dy, x, gam, m, r))
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


# Every general-form kernel (ring, register, element-wise), forced, on row
# lengths inside its capacity: several tiles per CTA and a ragged last tile
# (M prime), mixed types, strided rows, a residual add and dres.
def _force_cases():
    import rmsnorm_norm_fwd_gb300 as g
    cases = []
    for op in ("rms", "ln"):
        for d, dn in ((0, "fwd"), (1, "bwd")):
            for name in g.ex_variants(op == "ln", d):
                m = re.match(r"exr?[fb](\d+)x(\d+)b(\d+)", name)
                cap = int(m.group(1)) * int(m.group(2)) * 8 if m else 4096
                cases.append((op, dn, name, cap))
    return cases


def _cases_or_empty():
    try:
        return _force_cases()
    except Exception:  # library not built: collected as one skipped case
        return [("rms", "fwd", "unbuilt", 0)]


def _ring_fits(ln, d, name, M, N, xdt, ydt, pdt, extra):
    """Whether the planner may take ring kernel `name` for this call: a build
    for one row storage type only when x and y (dy) have it, and a ring
    layout that fits (about 16 KB of rows per stage, two stages per row group
    at least, in the opt-in shared memory after the header and the
    parameters)."""
    es = {"fp32": 4, "bf16": 2, "fp16": 2}
    m = re.fullmatch(r"exr[fb](\d+)x(\d+)b(\d+)(?:_(bf16|fp16|fp32))?", name)
    tpr, vpt, nt = (int(v) for v in m.groups()[:3])
    if m.group(4) and (m.group(4) != xdt or ydt != xdt):
        return False  # built for one row storage type shared by x and y / dy
    rpp = nt // tpr
    al = lambda b: (b + 127) // 128 * 128  # noqa: E731
    optin = torch.cuda.get_device_properties(0).shared_memory_per_block_optin
    budget = optin - 2048 - al(N * es[pdt]) * (2 if d == 0 and ln else 1)

    def stride(rt):
        st = al(rt * N * es[xdt]) * (2 if extra else 1)
        if d == 1:
            st += al(rt * N * es[ydt]) + al(((rt + 7) & ~3) * 4 * (2 if ln else 1))
        return st
    per_row = N * es[xdt] * (2 if extra else 1) + (N * es[ydt] if d == 1 else 0)
    rt = max(1, min(64, 16384 // per_row, M))
    while rt > 1 and 2 * rpp * stride(rt) > budget:
        rt //= 2
    if 2 * rpp * stride(rt) > budget:
        return False
    stages = min(16, budget // stride(rt))
    stages -= stages % rpp
    ring = stages * stride(rt)
    if d == 1 and rpp > 1:
        ring = max(ring, nt * vpt * 8 * 4 * (2 if ln else 1))
    return ring <= budget


@pytest.mark.parametrize("op,direction,name,cap", _cases_or_empty(),
                         ids=lambda v: str(v))
@pytest.mark.parametrize("types", [("bf16", "fp32", "bf16", True), ("fp32", "bf16", "fp16", False),
                                   ("fp16", "bf16", "fp16", True), ("fp32", "fp32", "fp32", False)],
                         ids=["bf16-fp32-extras", "fp32-bf16-fp16y", "fp16-bf16-extras", "fp32"])
def test_forced_variant(op, direction, name, cap, types):
    """Every general-form kernel, forced, at a row length inside its capacity,
    several tiles per CTA with a ragged last tile, against the oracle; a ring
    kernel whose layout cannot fit the call gives way to the usual choice."""
    import rmsnorm_norm_fwd_gb300 as g
    if name == "unbuilt":
        pytest.skip("library not built")
    ln = op == "ln"
    d = 0 if direction == "fwd" else 1
    xdt, pdt, ydt, extras = types
    N = cap if cap <= 4096 else cap - 8 * 37  # fills the capacity, or leaves part of it empty
    N = max(8, min(N, 16384))
    M = 389 if N <= 4096 else 41
    dist = "llm" if N >= 4096 else op
    inp = make_inputs(M, N, dtype=xdt, dist=dist, op=op, param_dtype=pdt, dy_dtype=ydt)
    res = make_inputs(M, N, dtype=xdt, dist="rms", op=op, seed=97).x if extras else None
    dres = make_inputs(M, N, dtype=xdt, dist="rms", op=op, seed=96).dy if extras else None
    g.ex_force_variant(ln, d, name)
    try:
        out, variants = run_ex(op, inp, pad=8, y_dtype=ydt, residual=res, dres=dres, check_path=False)
    finally:
        g.ex_force_variant(ln, d, None)
    served = name == "exe" or not name.startswith("exr") or _ring_fits(ln, d, name, M, N, xdt, ydt, pdt, extras)
    assert (variants[d] == name) == served, (variants, served)
    inp_h = make_inputs(M, N, dtype=xdt, dist=dist, op=op, param_dtype=pdt, dy_dtype=ydt)
    if extras:
        inp_h.x = oracle.residual_add(inp.x, res, xdt)
    compare(op, inp_h, out, variants=variants, y_dtype=ydt, dres=dres).assert_ok()

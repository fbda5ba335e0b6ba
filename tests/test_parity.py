"""CUDA path vs the fp64 oracle on small and ragged shapes, every variant,
and the edge cases (GPU; every call goes through the C ABI)."""
import re

import numpy as np
import pytest
import torch

from parity_util import compare, gpu_run, run_case
from rmsnorm_norm_fwd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

DTYPES = ["bf16", "fp16", "fp32"]
# Row lengths spanning every dispatch bucket, non-powers of two, and tails
# that do not fill a vector (element-wise path).
SMALL_N = [1, 3, 8, 63, 256, 384, 1000, 1024, 2048, 4096, 5120, 8192, 16392, 32768, 65536, 131072]


def _rows_for(N):
    # A few hundred rows for short rows (several CTAs and a ragged last
    # iteration), fewer for wide rows so that the oracle stays quick.
    return 301 if N <= 4096 else (37 if N <= 32768 else 9)


@pytest.mark.parametrize("N", SMALL_N)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", ["rms", "ln"])
def test_small_shapes(op, dtype, N):
    rep, _, _ = run_case(op, dtype, _rows_for(N), N, dist="llm" if N >= 4096 else None)
    rep.assert_ok()


def _geom(name):
    """(tpr, vpt, rows, cluster, cta, is_tma) of a vector variant, None for 'elem'."""
    if name.startswith("sk"):  # single-kernel backward: the staged kernel's geometry
        return _geom(name[2:])
    m = re.fullmatch(r"(\d+)x(\d+)r(\d+)c(\d+)b(\d+)", name)
    if m:
        return tuple(int(v) for v in m.groups()) + (False,)
    m = re.fullmatch(r"s(\d+)x(\d+)b(\d+)m(\d+)r?", name)
    if m:
        tpr, vpt, cta, _ = (int(v) for v in m.groups())
        return (tpr, vpt, 1, 1, cta, False)
    m = re.fullmatch(r"tmp(\d+)x(\d+)b(\d+)", name)
    if m:
        tpr, vpt, nt = (int(v) for v in m.groups())
        return (tpr, vpt, 1, 1, nt, True)
    m = re.fullmatch(r"tma(\d+)x(\d+)w(\d+)", name)
    if m:
        tpr, vpt, cw = (int(v) for v in m.groups())
        return (tpr, vpt, 1, 1, cw * 32, True)
    m = re.fullmatch(r"tmac(\d+)x(\d+)s(\d+)", name)
    if m:
        cl, vpt, rs = (int(v) for v in m.groups())
        return (256, vpt, rs, cl, 288, True)
    m = re.fullmatch(r"wide(\d+)u(\d+)b(\d+)p(\d+)r(\d+)", name)
    if m:
        nt, u, _, _, _ = (int(v) for v in m.groups())
        return ("wide", nt, u, 1)
    m = re.fullmatch(r"bwtma(\d+)x(\d+)", name)
    if m:
        cl, k = (int(v) for v in m.groups())
        return ("bwtma", 512, k, cl)
    m = re.fullmatch(r"wcs(\d+)v(\d+)c(\d+)", name)
    if m:
        nt, vpt, cl = (int(v) for v in m.groups())
        return ("wcs", nt, vpt, cl)
    m = re.fullmatch(r"bwr(\d+)k(\d+)c(\d+)p(\d+)m(\d+)f(\d+)[dg]?", name)
    if m:
        nt, k, cl, _, _, _ = (int(v) for v in m.groups())
        return ("bwtma", nt, k, cl)
    m = re.fullmatch(r"fwr(\d+)k(\d+)c(\d+)p(\d+)m(\d+)f(\d+)", name)
    if m:
        nt, k, cl, _, _, _ = (int(v) for v in m.groups())
        return ("bwtma", nt, k, cl)
    m = re.fullmatch(r"wtma(\d+)x(\d+)", name)
    if m:
        cw, u = (int(v) for v in m.groups())
        return ("wide", 32 * cw, u, 1)
    m = re.fullmatch(r"bwide(\d+)u(\d+)c(\d+)p(\d+)f(\d+)m(\d+)", name)
    if m:
        nt, u, cl, _, _, _ = (int(v) for v in m.groups())
        return ("wide", nt, u, cl)
    return None


@pytest.fixture(autouse=True)
def _no_device_fault():
    """Every test must leave the device fault word clear (no bounded wait gave up)."""
    import rmsnorm_norm_fwd_gb300 as g
    g.read_fault(reset=True)
    yield
    assert g.read_fault(reset=True) == 0, "a kernel's bounded wait timed out"


def _variant_cases():
    import rmsnorm_norm_fwd_gb300 as g
    cases = []
    for op in ("rms", "ln"):
        for d in (0, 1):
            for dt in DTYPES:
                for v in g.variants(op == "ln", d, dt):
                    cases.append((op, d, dt, v))
    return cases


def _variant_ids():
    try:
        return [f"{o}-{'fwd' if d == 0 else 'bwd'}-{t}-{v}" for o, d, t, v in _variant_cases()]
    except Exception:
        return None


try:
    _CASES = _variant_cases()
except Exception:  # library not built (collection on a machine without it)
    _CASES = []


@pytest.mark.parametrize("op,direction,dtype,variant", _CASES, ids=_variant_ids())
def test_forced_variant(op, direction, dtype, variant):
    """Each compiled variant, forced, at its full row capacity and at a row
    one vector short of it, with a ragged number of rows."""
    import rmsnorm_norm_fwd_gb300 as g
    E = 4 if dtype == "fp32" else 8
    geo = _geom(variant)
    if geo is None:  # the element-wise variant: odd N
        shapes = [(67, 1), (67, 77), (5, 3001)]
    elif geo[0] == "bwtma":
        # column slices of CL CTAs, K chunks of 512 vectors each: full slices,
        # one vector short, a ragged last chunk, and CTAs left without columns
        nt, k, cl = geo[1], geo[2], geo[3]
        cap = cl * k * nt * E
        shapes = [(9, cap), (9, cap - E), (7, cap // 2 + 3 * E), (5, cl * 3 * E), (3, (cl - 1) * E)]
    elif geo[0] == "wcs":
        # cluster slices resident in shared memory: full slices, one vector
        # short, a ragged last slice, three vectors per CTA
        nt, vpt, cl = geo[1], geo[2], geo[3]
        cap = cl * vpt * nt * E
        shapes = [(9, cap), (9, cap - E), (7, cap // 2 + 3 * E), (5, cl * 3 * E)]
    elif geo[0] == "wide":
        # any row length (per CTA of the cluster): two full load batches per
        # thread, one vector short of that, a slice where only part of the CTA
        # holds a last vector, and a slice shorter than the CTA (threads
        # without elements).  The backward keeps each slice's dgamma/dbeta
        # sums in shared memory: the widest rows that fit are taken.
        nt, u, cl = geo[1], geo[2], geo[3]
        full = cl * 2 * nt * u * E
        shapes = [(9, full), (9, full - E), (7, cl * (nt * E + 5 * E)), (5, cl * 3 * E)]
        if variant.startswith("wtma"):  # several ring jobs per pass, a ragged last one
            shapes.append((3, 7 * nt * u * E + 3 * E))
    else:
        tpr, vpt, r, cl, cta, tma = geo
        cap = tpr * vpt * cl * E
        if tma and cl > 1:
            M = 11  # a few rows per cluster; rows not a multiple of 4 (statistics tail)
        elif tma:
            # several tiles, a ragged last tile (not a multiple of 4 rows)
            M = max(7, min(1000, (3 << 20) // (cap * (4 if dtype == "fp32" else 2))) | 3)
        else:
            rows_per_iter = r if cl > 1 else (cta // tpr) * r
            M = min(2 * rows_per_iter + 3, max(3, (1 << 21) // cap))
        shapes = [(M, cap), (M, cap - E)]
    try:
        g.force_variant(op == "ln", direction, dtype, variant)
        if geo is not None and geo[0] == "bwtma":
            shapes = [(m, n) for m, n in shapes if n >= E]
        if geo is not None and geo[0] == "wide" and direction == 1:
            # the widest of the rows above whose slice sums fit
            full = shapes[0][1]
            while full > geo[3] * E and g.variant_name(op == "ln", 1, 9, full, dtype) != variant:
                full //= 2
            shapes = [(9, full), (9, full - E)] + shapes[2:]
        if geo is not None and geo[0] not in ("wide", "bwtma", "wcs") and geo[5]:
            # A staged variant may hold fewer elements than its register
            # capacity when gamma/beta and two stages must fit in shared
            # memory: take the widest row it serves, at least a quarter of it.
            M, cap = shapes[0]
            n = cap
            while n >= cap // 4 and g.variant_name(op == "ln", direction, M, n, dtype) != variant:
                n //= 2
            assert n >= cap // 4, f"{variant} serves no row of {cap // 4}..{cap} elements"
            shapes = [(M, n), (M, n - E)]
        for (M, N) in shapes:
            assert g.variant_name(op == "ln", direction, M, N, dtype, aligned=(geo is not None)) == variant
            rep, _, _ = run_case(op, dtype, M, N, dist="llm")
            rep.assert_ok()
    finally:
        g.force_variant(op == "ln", direction, dtype, None)


@pytest.mark.parametrize("op", ["rms", "ln"])
def test_empty_rows(op):
    import rmsnorm_norm_fwd_gb300 as g
    N = 256
    x = torch.empty(0, N, device="cuda", dtype=torch.bfloat16)
    gam = torch.ones(N, device="cuda", dtype=torch.bfloat16)
    dg = torch.full((N,), 7.0, device="cuda")
    db = torch.full((N,), 7.0, device="cuda")
    if op == "rms":
        y, r = g.rmsnorm_fwd(x, gam, 1e-6)
        dx, dg = g.rmsnorm_bwd(x, x, gam, r, dgamma=dg)
    else:
        y, m, r = g.layernorm_fwd(x, gam, gam, 1e-5)
        dx, dg, db = g.layernorm_bwd(x, x, gam, m, r, dgamma=dg, dbeta=db)
        assert torch.all(db == 0)
    torch.cuda.synchronize()
    assert y.shape == (0, N) and torch.all(dg == 0)


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_misaligned_pointers_take_the_elementwise_path(op, dtype):
    """Rows starting off a 16-byte boundary: the vector kernels must not be
    used, and results must still match."""
    M, N = 97, 1024
    inp = make_inputs(M, N, dtype=dtype, op=op)
    xb = torch.empty(M * N + 1, device="cuda", dtype=inp.x.dtype)
    db = torch.empty(M * N + 1, device="cuda", dtype=inp.x.dtype)
    x = xb[1:].view(M, N)
    dy = db[1:].view(M, N)
    x.copy_(inp.x)
    dy.copy_(inp.dy)
    assert x.data_ptr() % 16 != 0
    out = gpu_run(op, inp, x_dev=x, dy_dev=dy)
    compare(op, inp, out).assert_ok()


@pytest.mark.parametrize("op", ["rms", "ln"])
def test_in_place(op):
    import rmsnorm_norm_fwd_gb300 as g
    M, N = 129, 2048
    inp = make_inputs(M, N, op=op)
    ref = gpu_run(op, inp)
    x = inp.x.cuda()
    dy = inp.dy.cuda()
    gam, bet = inp.gamma.cuda(), inp.beta.cuda()
    if op == "rms":
        y, r = g.rmsnorm_fwd(x.clone(), gam, inp.eps)
        xi = x.clone()
        y2, _ = g.rmsnorm_fwd(xi, gam, inp.eps, y=xi)
        dyi = dy.clone()
        dx2, _ = g.rmsnorm_bwd(dyi, x, gam, r, dx=dyi)
    else:
        y, m, r = g.layernorm_fwd(x.clone(), gam, bet, inp.eps)
        xi = x.clone()
        y2, _, _ = g.layernorm_fwd(xi, gam, bet, inp.eps, y=xi)
        dyi = dy.clone()
        dx2, _, _ = g.layernorm_bwd(dyi, x, gam, m, r, dx=dyi)
    torch.cuda.synchronize()
    assert torch.equal(y2, ref["y"]) and torch.equal(dx2, ref["dx"])


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("N", [384, 8192, 65536])
def test_deterministic(op, N):
    M = 1024 if N <= 8192 else 64
    inp = make_inputs(M, N, op=op)
    a = gpu_run(op, inp)
    b = gpu_run(op, inp)
    for k in a:
        if k != "variants":
            assert torch.equal(a[k], b[k]), k


def test_rms_scale_equivariance():
    """x -> 2x with eps -> 4 eps leaves y unchanged and halves rstd (within
    tolerance: nothing is assumed about the device's rsqrt)."""
    import rmsnorm_norm_fwd_gb300 as g
    inp = make_inputs(512, 1024, dtype="fp32")
    x, gam = inp.x.cuda(), inp.gamma.cuda()
    y1, r1 = g.rmsnorm_fwd(x, gam, 1e-6)
    y2, r2 = g.rmsnorm_fwd(2 * x, gam, 4e-6)
    torch.cuda.synchronize()
    assert torch.allclose(y1, y2, rtol=1e-6, atol=1e-7)
    assert torch.allclose(r1, 2 * r2, rtol=1e-6)


def test_degenerate_rows():
    """Zero rows (RMS: y = 0, rstd = 1/sqrt(eps)) and constant rows (LN:
    y = beta) against the oracle."""
    M, N = 64, 512
    for op in ("rms", "ln"):
        for dtype in DTYPES:
            inp = make_inputs(M, N, dtype=dtype, op=op)
            inp.x[::2] = 0
            inp.x[1::4] = 1.5
            out = gpu_run(op, inp)
            compare(op, inp, out).assert_ok()


# A staged variant per (direction, N) that the ring-wrap test forces.
RING_VARIANTS = {(0, 256): "tma32x1w8", (1, 256): "tma16x2w8", (0, 2048): "tma32x8w8",
                 (1, 2048): "tma128x2w8", (0, 8192): "tma128x8w8", (1, 8192): "tma256x4w8",
                 (0, 65536): "tmac8x4s2", (1, 65536): "tmac8x4s2"}


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("direction", [0, 1])
@pytest.mark.parametrize("N", [256, 2048, 8192, 65536])
@pytest.mark.parametrize("limit", [1, 3])
def test_tma_ring_wraps(op, direction, N, limit):
    """A capped grid makes each CTA (or cluster) walk many more tiles than the
    ring has stages, so every stage's barriers -- and, for wide rows, the
    cluster's exchange barriers -- go through several phases.  For wide rows
    the cap is in CTAs: 8 and 24 CTAs leave one and three clusters."""
    import rmsnorm_norm_fwd_gb300 as g
    M = 4099 if N <= 2048 else (517 if N <= 8192 else 37)
    variant = RING_VARIANTS[(direction, N)]
    if N > 8192:
        limit = limit * 8
    try:
        g.force_variant(op == "ln", direction, "bf16", variant)
        g.set_grid_limit(limit)
        assert g.variant_name(op == "ln", direction, M, N, "bf16") == variant
        rep, _, _ = run_case(op, "bf16", M, N)
        rep.assert_ok()
    finally:
        g.set_grid_limit(0)
        g.force_variant(op == "ln", direction, "bf16", None)


# Wide-row variants (one CTA per row, or a cluster with an exchange ring of
# four slots) that the pipeline test forces, per (direction, N).
WIDE_PIPE = {(0, 16384): "wide512u8b2p1r1", (0, 65536): "wide1024u4b1p1r1", (0, 32768): "wide512u4b2p1r2",
             (1, 8192): "bwide512u4c1p1f0m1", (1, 16384): "bwide512u2c1p2f1m1",
             (1, 32768): "bwide512u2c2p2f1m1", (1, 32760): "bwide512u4c2p1f0m1",
             (1, 65536): "bwide512u2c4p2f1m1", (1, 65528): "bwide512u4c4p2f0m1",
             (1, 131072): "bwide512u2c8p2f1m1"}


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("key", sorted(WIDE_PIPE), ids=lambda k: f"{'fwd' if k[0] == 0 else 'bwd'}-{k[1]}")
@pytest.mark.parametrize("limit", [1, 3])
def test_wide_rows_pipeline(op, key, limit):
    """A capped grid gives each CTA (or cluster) many rows in turn: the
    forward's prefetch chain and the backward's pipeline (pass 2 two rows
    behind pass 1, exchange barriers and slots reused every fourth row) run
    through every phase, including rows counts that are not multiples of 4."""
    import rmsnorm_norm_fwd_gb300 as g
    direction, N = key
    variant = WIDE_PIPE[key]
    cl = int(re.search(r"c(\d+)p", variant).group(1)) if variant.startswith("bwide") else 1
    M = 23
    try:
        g.force_variant(op == "ln", direction, "bf16", variant)
        if g.variant_name(op == "ln", direction, M, N, "bf16") != variant:
            pytest.skip(f"{variant} cannot hold {op} rows of {N}")
        g.set_grid_limit(limit * cl)
        assert g.variant_name(op == "ln", direction, M, N, "bf16") == variant
        rep, _, _ = run_case(op, "bf16", M, N)
        rep.assert_ok()
    finally:
        g.set_grid_limit(0)
        g.force_variant(op == "ln", direction, "bf16", None)


def test_grid_limit_changes_nothing():
    import rmsnorm_norm_fwd_gb300 as g
    inp = make_inputs(3001, 768, op="ln", dist="ln")
    a = gpu_run("ln", inp)
    try:
        g.set_grid_limit(5)
        b = gpu_run("ln", inp)
    finally:
        g.set_grid_limit(0)
    for k in ("y", "mean", "rstd", "dx"):
        assert torch.equal(a[k], b[k]), k
    # dgamma/dbeta are summed in a different grouping: equal within tolerance
    for k in ("dgamma", "dbeta"):
        assert torch.allclose(a[k], b[k], rtol=1e-5, atol=1e-4), k


def test_unaligned_stats_fall_back_from_tma():
    """rstd/mean not 16-byte aligned: the backward must not use the bulk-copy
    kernels (which copy them in 16-byte units) and must still be right."""
    import rmsnorm_norm_fwd_gb300 as g
    M, N = 1029, 1024
    inp = make_inputs(M, N, op="ln", dist="ln")
    x, dy = inp.x.cuda(), inp.dy.cuda()
    gam, bet = inp.gamma.cuda(), inp.beta.cuda()
    y, mean, rstd = g.layernorm_fwd(x, gam, bet, inp.eps)
    mb = torch.empty(M + 1, device="cuda")
    rb = torch.empty(M + 1, device="cuda")
    mean_u, rstd_u = mb[1:], rb[1:]
    mean_u.copy_(mean)
    rstd_u.copy_(rstd)
    assert rstd_u.data_ptr() % 16 != 0
    dx, dg, db = g.layernorm_bwd(dy, x, gam, mean_u, rstd_u)
    torch.cuda.synchronize()
    out = {"y": y, "mean": mean, "rstd": rstd, "dx": dx, "dgamma": dg, "dbeta": db}
    # the backward that ran is not the one aligned statistics select: take the
    # deeper of the two sums
    vf = g.variant_name(True, 0, M, N, "bf16")
    vb = [g.variant_name(True, 1, M, N, "bf16"), g.variant_name(True, 1, M, N, "bf16", aligned=False)]
    compare("ln", inp, out, variants=(vf, vb)).assert_ok()


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N", [1000, 4096, 65536])
def test_optional_parameters(op, dtype, N):
    """A NULL gamma (and beta) reads gamma = 1 (beta = 0), against the oracle
    with those rows; a dgamma / dbeta not asked for is not produced and leaves
    dx and the other sum unchanged (bitwise)."""
    import rmsnorm_norm_fwd_gb300 as g
    M = 37 if N <= 4096 else 9
    inp = make_inputs(M, N, dtype=dtype, dist="llm" if N >= 4096 else op, op=op)
    inp.gamma = torch.ones_like(inp.gamma)
    inp.beta = torch.zeros_like(inp.beta)
    x, dy = inp.x.cuda(), inp.dy.cuda()
    if op == "rms":
        y, rstd = g.rmsnorm_fwd(x, None, inp.eps)
        dx, dgam = g.rmsnorm_bwd(dy, x, None, rstd, need_dgamma=False)
        assert dgam is None
        dx2, dgam2 = g.rmsnorm_bwd(dy, x, None, rstd)
        out = dict(y=y, rstd=rstd, dx=dx, dgamma=dgam2)
    else:
        y, mean, rstd = g.layernorm_fwd(x, None, None, inp.eps)
        dx, dgam, dbet = g.layernorm_bwd(dy, x, None, mean, rstd, need_dgamma=False)
        assert dgam is None and dbet is not None
        dx2, dgam2, dbet2 = g.layernorm_bwd(dy, x, None, mean, rstd, need_dbeta=False)
        assert dbet2 is None
        out = dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dgam2, dbeta=dbet)
    torch.cuda.synchronize()
    assert torch.equal(dx, dx2)
    compare(op, inp, out).assert_ok()


# Single-kernel backward variants, each against the two-kernel variant of the
# same geometry: (op, variant, dtype, M, N).
SK_CASES = [("rms", "sktma32x4w8", "bf16", 1024, 1024), ("ln", "sktma32x4w8", "bf16", 1024, 1024),
            ("rms", "sktma16x2w8", "bf16", 1001, 256), ("ln", "sktma128x4w8", "fp32", 300, 2048),
            ("rms", "sktma256x8w8", "bf16", 200, 16384), ("ln", "sktmp256x4b512", "bf16", 513, 8192),
            ("rms", "sktmp128x4b512", "fp16", 77, 4096), ("ln", "sktmp512x4b512", "fp32", 129, 8192)]


@pytest.mark.parametrize("op,variant,dtype,M,N", SK_CASES, ids=[f"{c[0]}-{c[1]}-{c[2]}-{c[3]}x{c[4]}" for c in SK_CASES])
@pytest.mark.parametrize("limit", [0, 1, 5])
def test_single_kernel_backward(op, variant, dtype, M, N, limit):
    """The single-kernel backward (cooperative launch; the kernel sums the
    partial rows itself once every CTA's flag carries the call's epoch) gives
    dx, dgamma and dbeta bit-identical to the two-kernel path with the same
    grid, twice in a row on one workspace (the second call meets the first
    call's flags), under a grid cap (several tiles per CTA; one CTA alone),
    with a sum not asked for, and within tolerance of the oracle."""
    import rmsnorm_norm_fwd_gb300 as g
    ln = op == "ln"
    inp = make_inputs(M, N, dtype=dtype, dist="llm" if N >= 4096 else op, op=op)
    x, dy, gam, bet = (t.cuda() for t in (inp.x, inp.dy, inp.gamma, inp.beta))
    if ln:
        y, mean, rstd = g.layernorm_fwd(x, gam, bet, inp.eps)
    else:
        (y, rstd), mean = g.rmsnorm_fwd(x, gam, inp.eps), None

    def bwd(ws, **kw):
        if ln:
            return g.layernorm_bwd(dy, x, gam, mean, rstd, workspace=ws, **kw)
        return g.rmsnorm_bwd(dy, x, gam, rstd, workspace=ws, **kw)

    runs = {}
    try:
        g.set_grid_limit(limit)
        for v in (variant[2:], variant):
            g.force_variant(ln, 1, dtype, v)
            assert g.variant_name(ln, 1, M, N, dtype) == v
            ws = torch.empty(g.norm_bwd_workspace_size(ln, M, N, dtype), device="cuda", dtype=torch.uint8)
            runs[v] = [bwd(ws), bwd(ws)]
            if ln:
                runs[v].append(bwd(ws, need_dgamma=False))
        torch.cuda.synchronize()
    finally:
        g.set_grid_limit(0)
        g.force_variant(ln, 1, dtype, None)
    ref = runs[variant[2:]][0]
    for got in runs[variant][:2] + runs[variant[2:]][1:2]:
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
    if ln:  # dbeta alone, dgamma not produced: the same dx and dbeta
        dx3, dg3, db3 = runs[variant][2]
        assert dg3 is None and torch.equal(dx3, ref[0]) and torch.equal(db3, ref[2])
    out = {"y": y, "rstd": rstd, "dx": ref[0], "dgamma": ref[1]}
    if ln:
        out.update(mean=mean, dbeta=ref[2])
    compare(op, inp, out, variants=(g.variant_name(ln, 0, M, N, dtype), variant)).assert_ok()


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("variant", ["wtma16x2", "wtma8x2"])
@pytest.mark.parametrize("limit", [1, 3])
def test_wide_ring_wraps(op, variant, limit):
    """The bulk-copy wide forward under a grid cap: each CTA walks many rows,
    so every ring stage goes through many phases, with pass-1 and pass-2 jobs
    of different sizes interleaved (row length not a multiple of a chunk)."""
    import rmsnorm_norm_fwd_gb300 as g
    M, N = 23, 3 * 8192 + 40
    try:
        g.force_variant(op == "ln", 0, "bf16", variant)
        g.set_grid_limit(limit)
        assert g.variant_name(op == "ln", 0, M, N, "bf16") == variant
        rep, _, _ = run_case(op, "bf16", M, N)
        rep.assert_ok()
    finally:
        g.set_grid_limit(0)
        g.force_variant(op == "ln", 0, "bf16", None)


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("direction", [0, 1])
@pytest.mark.parametrize("variant,N", [("wcs512v4c8", 131072), ("wcs512v2c16", 131072 - 24),
                                       ("wcs512v4c4", 65536 - 8 * 5), ("wcs512v4c8", 3000)])
@pytest.mark.parametrize("limit", [1, 3])
def test_wcs_ring_wraps(op, direction, variant, N, limit):
    """The cluster kernels with row slices resident in shared memory, under a
    grid cap (in clusters): each cluster walks many rows, so the ring stages
    (refilled as each row's pass 2 ends), the pass order (pass 1 one row
    ahead) and the four exchange slots go through many phases."""
    import rmsnorm_norm_fwd_gb300 as g
    cl = int(re.search(r"c(\d+)$", variant).group(1))
    M = 29
    try:
        g.force_variant(op == "ln", direction, "bf16", variant)
        g.set_grid_limit(limit * cl)
        assert g.variant_name(op == "ln", direction, M, N, "bf16") == variant
        rep, _, _ = run_case(op, "bf16", M, N)
        rep.assert_ok()
    finally:
        g.set_grid_limit(0)
        g.force_variant(op == "ln", direction, "bf16", None)


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("variant,N", [("fwr256k8c8p1m2f0", 131072), ("fwr256k8c4p0m2f0", 65536 - 24),
                                       ("fwr512k4c2p0m1f0", 32768 - 8), ("fwr256k8c1p0m2f0", 16384),
                                       ("fwr256k4c16p0m2f0", 131072 - 8 * 9), ("fwr256k8c8p0m2f1", 131072),
                                       ("fwr256k8c4p0m2f1", 65536 - 8 * 3), ("fwr256k8c8p0m2f2", 131072),
                                       ("fwr256k8c4p0m2f2", 65536 - 24), ("fwr512k8c1p0m1f2", 32768 - 8 * 9),
                                       ("fwr256k8c1p0m2f2", 16384 - 8), ("fwr256k4c1p0m4f2", 8192),
                                       ("fwr256k8c2p0m2f2", 32768 - 8)])
@pytest.mark.parametrize("limit", [1, 3])
def test_wide_forward_cluster_rows(op, variant, N, limit):
    """The cluster-slice wide forward under a grid cap (in clusters): each
    cluster walks many rows, so the four exchange slots and the pass order
    (pass 1 one row ahead of pass 2; in the one-pass form the two register
    buffers, with an odd row count ending on the first) go through many
    phases."""
    import rmsnorm_norm_fwd_gb300 as g
    cl = int(re.search(r"c(\d+)p", variant).group(1))
    M = 23
    try:
        g.force_variant(op == "ln", 0, "bf16", variant)
        g.set_grid_limit(limit * cl)
        assert g.variant_name(op == "ln", 0, M, N, "bf16") == variant
        rep, _, _ = run_case(op, "bf16", M, N)
        rep.assert_ok()
    finally:
        g.set_grid_limit(0)
        g.force_variant(op == "ln", 0, "bf16", None)


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("variant,N", [("bwtma8x4", 131072), ("bwtma4x4", 65536 - 24), ("bwtma8x2", 40000),
                                       ("bwr512k4c8p1m1f1", 131072), ("bwr512k8c4p1m1f0", 131072 - 24),
                                       ("bwr256k4c16p1m2f1", 131072), ("bwr256k8c8p1m2f0", 131072 - 24),
                                       ("bwr256k4c2p1m2f1", 3000), ("bwr512k4c1p1m1f1", 16384),
                                       ("bwr512k4c1p1m1f0", 16384), ("bwr256k8c8p1m2f0d", 131072),
                                       ("bwr256k8c8p1m2f1d", 131072 - 24), ("bwr512k8c4p1m1f0d", 65536 + 8),
                                       ("bwr256k8c8p1m2f0g", 131072 - 24), ("bwr256k8c4p1m2f0g", 65536)])
@pytest.mark.parametrize("limit", [1, 3])
def test_wide_backward_ring_wraps(op, variant, N, limit):
    """The bulk-copy wide backward under a grid cap (in clusters): each cluster
    walks many rows, so the ring stages, the pass order (pass 1 one row ahead
    of pass 2) and the four exchange slots go through many phases."""
    import rmsnorm_norm_fwd_gb300 as g
    if variant.endswith(("d", "g")) and op != "ln":
        pytest.skip("dbeta-in-shared-memory variants exist for LayerNorm only")
    cl = int(re.match(r"bwtma(\d+)x", variant).group(1)) if variant.startswith("bwtma") else \
        int(re.search(r"c(\d+)p", variant).group(1))
    M = 23
    try:
        g.force_variant(op == "ln", 1, "bf16", variant)
        g.set_grid_limit(limit * cl)
        assert g.variant_name(op == "ln", 1, M, N, "bf16") == variant
        rep, _, _ = run_case(op, "bf16", M, N)
        rep.assert_ok()
    finally:
        g.set_grid_limit(0)
        g.force_variant(op == "ln", 1, "bf16", None)

"""GPU-vs-oracle comparison with the stated tolerances.

Both sides read the same seeded host tensors (``rmsnorm_norm_fwd_gb300.inputs``).
The GPU side goes through the Python binding, i.e. the C ABI; the oracle is
the fp64 C implementation in ``oracle/``.

Every bound below is computed from the oracle's values and from a-priori
constants of fp32 arithmetic only; nothing measured on the GPU output enters a
bound.  u = 2^-24 is the unit roundoff of fp32; ulp_T(v) is the spacing of
dtype T at |v| with v first rounded to T (the smallest subnormal spacing at 0).

Stated tolerances (the target figures for this path) and how they are read:
  y      : 1 ulp_T of the oracle value (fp16 also 2e-3 relative);
  rstd   : 1e-5 relative; mean: 1e-5 (|mean| + sigma);
  dx     : 2 ulp_T of the oracle value;
  dgamma, dbeta : ||d||_2 <= 1e-3 ||ref||_2.

No fp32 computation can meet a bare ulp bound where its result cancels
(y = xhat gamma + beta near 0, dx = rstd (g - c1 - xhat c2) near 0), so each
per-element bound adds the first-order error of the fp32 arithmetic that
produces it:

  D      : summation depth of a row sum in the kernel that ran, from its
           geometry (``sum_depth``): elements one thread adds serially
           (ceil(vectors / threads per row) * E), plus the levels that combine
           threads (log2 of the lanes of a warp, the warps of a row group in
           order, the CTAs of a cluster in order), plus 4.  A fp32 sum of n
           terms along a tree of depth D errs by at most D u sum|terms|.
  e_r    : a-priori relative error of the saved rstd, from the forward's D_f:
           RMS  u (D_f/2 + 7)  (sum of squares, divide, add eps, and rsqrtf's
           documented 2-ulp maximum error);
           LN   u (D_f/2 + 8) + u D_f rms(x) sigma / (var + eps)  (the second
           term: first-order error of the threads' and warps' means inside
           the exact (mean, M2) group combine; zero for the two-pass form);
  e_mu   : a-priori error of the saved mean: u (D_f + 2) mean|x|.

  y bound  = core_y + 4u (|xhat gamma| + |beta|) + |gamma| (rstd e_mu + |xhat| e_r)
             core_y = ulp_T(y_ref) (bf16, fp16: max with 2e-3|y_ref|); 0 for
             fp32 output (the fp32 result is the output).
  dx bound = 2 ulp_T(dx_ref)
             + u rstd (8 (|g| + |c1| + |xhat c2|)          final operations
                       + (D_b + 4) (|xhat| S2 + S1))        the row sums c2, c1
             + e_r (|dx_ref| + 2 rstd |xhat c2|)            saved rstd
             + rstd^2 e_mu (|c2| + |xhat c1|)               saved mean (LN)
           with g = dy gamma, S2 = (1/N) sum|g xhat|, S1 = (1/N) sum|g| (LN; 0
           for RMS), c2 = (1/N) sum g xhat, c1 = (1/N) sum g.
  rstd, mean are also held to e_r and e_mu, which the y and dx bounds assume.

Every check reports the largest error in output ulps and, for y and dx, how
many elements pass only through the floor terms (error above the bare 1-ulp /
2-ulp figure), so the fp32 behaviour is visible, not only pass/fail.  With
GBNORM_PARITY_LOG set to a path, every report's figures are appended there as
one JSON line per check.
"""
from __future__ import annotations

import json
import math
import os
import re
from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
from rmsnorm_norm_fwd_gb300.inputs import DTYPES, make_inputs

MANT = {"bf16": 7, "fp16": 10, "fp32": 23}
EMIN = {"bf16": -126, "fp16": -14, "fp32": -126}
ESIZE = {"bf16": 2, "fp16": 2, "fp32": 4}
U32 = 2.0 ** -24
RSQRT_ULPS = 2  # maximum error of rsqrtf (CUDA math API documentation)


def ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of `dtype` at |rnd_dtype(v)|."""
    r = torch.from_numpy(np.ascontiguousarray(v)).to(DTYPES[dtype]).double().numpy()
    a = np.abs(r)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, EMIN[dtype])
    u = np.exp2(e - MANT[dtype])
    u[a == 0] = 2.0 ** (EMIN[dtype] - MANT[dtype])
    return u


# ---------------------------------------------------------------- kernel geometry -> summation depth
def row_threads(variant: str):
    """(threads of one CTA that share a row, CTAs per row, element-wise?) of a
    compiled variant, from its name."""
    pats = (
        (r"(\d+)x(\d+)r(\d+)c(\d+)b(\d+)", lambda g: (g[0], g[3])),   # register rows (cluster)
        (r"s(\d+)x(\d+)b(\d+)m(\d+)r?", lambda g: (g[0], 1)),         # register rows, params in smem
        (r"tmp(\d+)x(\d+)b(\d+)", lambda g: (g[0], 1)),               # staged rows, no producer
        (r"tma(\d+)x(\d+)w(\d+)", lambda g: (g[0], 1)),               # staged rows, producer warp
        (r"tmac(\d+)x(\d+)s(\d+)", lambda g: (256, g[0])),            # staged cluster rows
        (r"wide(\d+)u(\d+)b(\d+)p(\d+)r(\d+)", lambda g: (g[0], 1)),  # wide forward
        (r"bwide(\d+)u(\d+)c(\d+)p(\d+)f(\d+)m(\d+)", lambda g: (g[0], g[2])),  # wide backward
        (r"wtma(\d+)x(\d+)", lambda g: (32 * g[0], 1)),             # wide forward, bulk-copy ring
        (r"bwtma(\d+)x(\d+)", lambda g: (512, g[0])),               # wide backward, bulk-copy ring
        (r"bwr(\d+)k(\d+)c(\d+)p(\d+)m(\d+)f(\d+)[dg]?", lambda g: (g[0], g[2])),  # wide bwd, register sums
        (r"wcs(\d+)v(\d+)c(\d+)", lambda g: (g[0], g[2])),           # cluster slices in shared memory
        (r"fwr(\d+)k(\d+)c(\d+)p(\d+)m(\d+)f(\d+)", lambda g: (g[0], g[2])),  # wide fwd, cluster slices
    )
    if variant.startswith("sk"):  # single-kernel backward: the staged kernel's geometry
        variant = variant[2:]
    m = re.fullmatch(r"exr?[fb](\d+)x(\d+)b(\d+)(?:_(?:bf16|fp16|fp32))?", variant)  # general form
    if m:
        return int(m.group(1)), 1, False
    for pat, f in pats:
        m = re.fullmatch(pat, variant)
        if m:
            tpr, cl = f([int(v) for v in m.groups()])
            return tpr, cl, False
    if variant in ("elem", "exe"):
        return 256, 1, True
    raise ValueError(f"unknown variant {variant!r}")


def sum_depth(N: int, variant: str, dtype: str) -> int:
    """Upper bound on the number of fp32 additions any term of a row sum passes
    through in `variant` (see the module docstring)."""
    tpr, cl, elem = row_threads(variant)
    E = 8 if variant.startswith("ex") else 16 // ESIZE[dtype]
    if elem:
        serial = -(-N // tpr)
    else:
        nv = -(-N // E)
        serial = -(-(-(-nv // cl)) // tpr) * E
    lanes = min(tpr, 32)
    tree = int(math.ceil(math.log2(lanes))) if lanes > 1 else 0
    tree += tpr // 32 if tpr > 32 else 0
    tree += cl if cl > 1 else 0
    return serial + tree + 4


# ---------------------------------------------------------------- bounds (oracle values only)
def apriori_stats(op, xn, rstd_ref, var_ref, eps, d_fwd):
    """(e_r, e_mu) per row: a-priori relative rstd error and absolute mean error."""
    base = RSQRT_ULPS * 2 + 3
    if op == "rms":
        e_r = U32 * (d_fwd / 2 + base) * np.ones(xn.shape[0])
        return e_r, np.zeros(xn.shape[0])
    mabs = np.abs(xn).mean(axis=1)
    rms = np.sqrt((xn * xn).mean(axis=1))
    sd = np.sqrt(np.maximum(var_ref, 0.0))
    e_r = U32 * (d_fwd / 2 + base + 1 + d_fwd * rms * sd / (var_ref + eps))
    e_mu = U32 * (d_fwd + 2) * mabs
    return e_r, e_mu


def y_bound(y_ref, xg_abs, beta_abs, dtype, gam_abs, xhat_abs, rstd, e_r, e_mu):
    arith = 4 * U32 * (xg_abs + beta_abs) + \
        gam_abs[None, :] * (rstd[:, None] * e_mu[:, None] + xhat_abs * e_r[:, None])
    if dtype == "fp32":
        return arith
    core = ulp(y_ref, dtype)
    if dtype == "fp16":
        core = np.maximum(core, 2e-3 * np.abs(y_ref))
    return core + arith


def dx_bound(dx_ref, rstd, g, c1, xhat, c2, s1, s2, e_r, e_mu, d_bwd, dtype, dres_abs=0.0):
    r = rstd[:, None]
    terms = np.abs(g) + np.abs(c1)[:, None] + np.abs(xhat * c2[:, None])
    arith = U32 * r * (8 * terms + (d_bwd + 4) * (np.abs(xhat) * s2[:, None] + s1[:, None])) + \
        2 * U32 * dres_abs
    stats = e_r[:, None] * (np.abs(dx_ref) + 2 * r * np.abs(xhat * c2[:, None])) + \
        r * r * e_mu[:, None] * (np.abs(c2)[:, None] + np.abs(xhat * c1[:, None]))
    return 2 * ulp(dx_ref, dtype) + arith + stats


# ---------------------------------------------------------------- report
@dataclass
class Report:
    ok: bool = True
    msgs: list = field(default_factory=list)
    stats: dict = field(default_factory=dict)
    case: dict = field(default_factory=dict)

    def check_elem(self, name, got, ref, bound, dtype=None, core_ulps=None, scale=None):
        """|got - ref| <= bound element-wise.  With dtype: also the largest
        error in ulps of dtype at ref, (core_ulps) how many elements are above
        core_ulps ulps, i.e. pass only through the floor terms, and (scale)
        the largest error in ulps of dtype at `scale`, the size of the terms
        that cancel into ref (the measure that stays meaningful where ref is
        near zero)."""
        err = np.abs(got.astype(np.float64) - ref)
        bad = ~(err <= bound)  # NaN counts as bad
        st = {"max_err": float(np.nanmax(err)) if err.size else 0.0,
              "max_err_over_bound": float(np.nanmax(err / np.maximum(bound, 1e-300))) if err.size else 0.0,
              "n_bad": int(bad.sum()), "n": int(err.size)}
        if dtype is not None and err.size:
            ue = err / ulp(ref, dtype)
            st["max_ulps"] = float(np.nanmax(ue))
            if core_ulps is not None:
                st["n_floor_only"] = int(((ue > core_ulps) & ~bad).sum())
            if scale is not None:
                st["max_ulps_of_terms"] = float(np.nanmax(err / ulp(scale, dtype)))
        self.stats[name] = st
        if bad.any():
            self.ok = False
            i = np.unravel_index(np.argmax(np.where(bad, err / np.maximum(bound, 1e-300), -1)), err.shape)
            self.msgs.append(f"{name}: {int(bad.sum())}/{err.size} out of bound; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} bound {bound[i]!r}")

    def check_l2(self, name, got, ref, rel=1e-3):
        d = np.linalg.norm(got.astype(np.float64) - ref)
        n = np.linalg.norm(ref)
        self.stats[name] = {"rel_l2": float(d / n) if n > 0 else float(d)}
        if not (d <= rel * n + 1e-30):
            self.ok = False
            self.msgs.append(f"{name}: relative L2 error {d / max(n, 1e-300):.3e} > {rel}")

    def check_equal(self, name, got, ref):
        same = torch.equal(got, ref)
        self.stats[name] = {"bitwise_equal": bool(same)}
        if not same:
            self.ok = False
            self.msgs.append(f"{name}: not bitwise equal")

    def log(self):
        path = os.environ.get("GBNORM_PARITY_LOG")
        if not path:
            return
        test = os.environ.get("PYTEST_CURRENT_TEST", "")
        with open(path, "a") as f:
            for k, v in self.stats.items():
                f.write(json.dumps({"test": test, **self.case, "check": k, **v}) + "\n")

    def summary(self) -> str:
        s = self.stats
        parts = []
        for k in ("y", "dx"):
            if k in s and "max_ulps" in s[k]:
                parts.append(f"{k} max {s[k]['max_ulps']:.2f} ulp ({s[k]['max_ulps_of_terms']:.2f} ulp of "
                             f"the terms), {s[k].get('n_floor_only', 0)} floor-only of {s[k]['n']}, "
                             f"err/bound {s[k]['max_err_over_bound']:.3f}")
        for k in ("dgamma", "dbeta"):
            if k in s:
                parts.append(f"{k} rel L2 {s[k]['rel_l2']:.2e}")
        return "; ".join(parts)

    def assert_ok(self):
        self.log()
        assert self.ok, "; ".join(self.msgs)


def _np(t):
    return t.detach().to("cpu").double().numpy()


def _aligned(*ts):
    return all(t is None or t.data_ptr() % 16 == 0 for t in ts)


def gpu_run(op, inp, device="cuda", x_dev=None, dy_dev=None):
    """Forward and backward on the GPU through the binding; returns host-side
    tensors plus the names of the variants that ran ('variants')."""
    import rmsnorm_norm_fwd_gb300 as g
    x = inp.x.to(device) if x_dev is None else x_dev
    dy = inp.dy.to(device) if dy_dev is None else dy_dev
    gamma = inp.gamma.to(device)
    beta = inp.beta.to(device)
    out = {}
    M, N = x.shape
    if op == "rms":
        y, rstd = g.rmsnorm_fwd(x, gamma, inp.eps)
        dx, dgam = g.rmsnorm_bwd(dy, x, gamma, rstd)
        out.update(y=y, rstd=rstd, dx=dx, dgamma=dgam)
    else:
        y, mean, rstd = g.layernorm_fwd(x, gamma, beta, inp.eps)
        dx, dgam, dbet = g.layernorm_bwd(dy, x, gamma, mean, rstd)
        out.update(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dgam, dbeta=dbet)
    torch.cuda.synchronize()
    ln = op == "ln"
    a_f = _aligned(x, y, gamma, beta if ln else None)
    a_b = _aligned(dy, x, out["dx"], gamma, rstd, out.get("mean"))
    out["variants"] = (g.variant_name(ln, 0, M, N, inp.dtype, aligned=a_f),
                       g.variant_name(ln, 1, M, N, inp.dtype, aligned=a_b))
    return out


def compare(op, inp, out, rows=None, variants=None, y_dtype=None, dres=None) -> Report:
    """Compare GPU outputs against the oracle.  rows=None: every row; else the
    listed rows for y/stats/dx (dgamma/dbeta always over all rows).
    variants: (forward, backward) names, or lists of names whose largest
    summation depth is taken; default out['variants'].  inp.x are the rows
    that were normalised (h after a residual add); y is held to y_dtype
    (default inp.dtype), dx to inp.dtype; dres (the gradient added into dx)
    enters the oracle's dx and, through its final fp32 add, the dx bound."""
    import rmsnorm_norm_fwd_gb300 as g
    rep = Report()
    dt = inp.dtype
    ydt = y_dtype or dt
    M, N = inp.x.shape
    if variants is None:
        variants = out.get("variants")
    if variants is None:
        ln = op == "ln"
        variants = (g.variant_name(ln, 0, M, N, dt), g.variant_name(ln, 1, M, N, dt))
    vf, vb = ([v] if isinstance(v, str) else list(v) for v in variants)
    d_fwd = max(sum_depth(N, v, dt) for v in vf)
    d_bwd = max(sum_depth(N, v, dt) for v in vb)
    rep.case = {"op": op, "dtype": dt, "y_dtype": ydt, "M": M, "N": N, "dist": inp.dist, "fwd": vf, "bwd": vb,
                "D_f": d_fwd, "D_b": d_bwd, "rows": None if rows is None else len(rows),
                "residual": dres is not None}
    x = inp.x if rows is None else inp.x[rows]
    dy = inp.dy if rows is None else inp.dy[rows]
    dr = None if dres is None else (dres if rows is None else dres[rows])
    sel = (lambda t: t) if rows is None else (lambda t: t[rows])
    gam = _np(inp.gamma)
    bet = _np(inp.beta) if op == "ln" else np.zeros_like(gam)
    if op == "rms":
        y_ref, rstd_ref = oracle.rmsnorm_fwd(x, inp.gamma, inp.eps)
        mean_ref = np.zeros_like(rstd_ref)
        dx_ref, _ = oracle.rmsnorm_bwd(dy, x, inp.gamma, inp.eps, want_dgamma=False, dres=dr)
        _, dg_ref = oracle.rmsnorm_bwd(inp.dy, inp.x, inp.gamma, inp.eps, want_dx=False)
        db_ref = None
    else:
        y_ref, mean_ref, rstd_ref = oracle.layernorm_fwd(x, inp.gamma, inp.beta, inp.eps)
        dx_ref, _, _ = oracle.layernorm_bwd(dy, x, inp.gamma, inp.eps, want_dparams=False, dres=dr)
        _, dg_ref, db_ref = oracle.layernorm_bwd(inp.dy, inp.x, inp.gamma, inp.eps, want_dx=False)
    xn = _np(x)
    var_ref = 1.0 / rstd_ref ** 2 - inp.eps
    xhat = (xn - mean_ref[:, None]) * rstd_ref[:, None]
    zeros = np.zeros(xn.shape[0])
    e_r, e_mu = apriori_stats(op, xn, rstd_ref, var_ref, inp.eps, d_fwd)
    rep.check_elem("y", _np(sel(out["y"])), y_ref,
                   y_bound(y_ref, np.abs(xhat * gam), np.abs(bet), ydt, np.abs(gam), np.abs(xhat),
                           rstd_ref, e_r, e_mu), dtype=ydt, core_ulps=1,
                   scale=np.abs(xhat * gam) + np.abs(bet))
    rstd_got = _np(sel(out["rstd"]))
    rep.check_elem("rstd", rstd_got, rstd_ref, 1e-5 * rstd_ref)
    rep.check_elem("rstd_apriori", rstd_got, rstd_ref, e_r * rstd_ref)
    if op == "ln":
        sd = np.sqrt(np.maximum(var_ref, 0.0))
        mean_got = _np(sel(out["mean"]))
        rep.check_elem("mean", mean_got, mean_ref, 1e-5 * (np.abs(mean_ref) + sd))
        rep.check_elem("mean_apriori", mean_got, mean_ref, e_mu + 1e-300)
    g_ = _np(dy) * gam
    c1 = g_.sum(axis=1) / N if op == "ln" else zeros
    c2 = (g_ * xhat).sum(axis=1) / N
    s1 = np.abs(g_).sum(axis=1) / N if op == "ln" else zeros
    s2 = np.abs(g_ * xhat).sum(axis=1) / N
    dra = 0.0 if dr is None else np.abs(_np(dr))
    rep.check_elem("dx", _np(sel(out["dx"])), dx_ref,
                   dx_bound(dx_ref, rstd_ref, g_, c1, xhat, c2, s1, s2, e_r, e_mu, d_bwd, dt, dra),
                   dtype=dt, core_ulps=2,
                   scale=rstd_ref[:, None] * (np.abs(g_) + np.abs(c1)[:, None] + np.abs(xhat * c2[:, None]))
                   + dra)
    rep.check_l2("dgamma", _np(out["dgamma"]), dg_ref)
    if op == "ln":
        rep.check_l2("dbeta", _np(out["dbeta"]), db_ref)
    return rep


def sample_rows(M: int, k: int = 62, seed: int = 5, x=None) -> np.ndarray:
    """First, last and k seeded rows; with x given, also every row whose root
    mean square exceeds 20 (the rows the accumulation-stress recipe scales by
    100), so that those rows are checked at every size."""
    rng = np.random.default_rng(seed)
    r = set(rng.choice(M, size=min(k, M), replace=False).tolist()) | {0, M - 1}
    if x is not None and M > 0:
        xs = x.float()
        ms = (xs * xs).mean(dim=1)
        r |= set(torch.nonzero(ms > 400.0).flatten().tolist())
    return np.array(sorted(r), dtype=np.int64)


def run_case(op, dtype, M, N, dist=None, rows=None, seed=None):
    """rows: None (every row), 'sample' (sample_rows with the stress rows), or
    an explicit index array."""
    kw = {} if seed is None else {"seed": seed}
    inp = make_inputs(M, N, dtype=dtype, dist=dist or ("ln" if op == "ln" else "rms"), op=op, **kw)
    out = gpu_run(op, inp)
    if isinstance(rows, str) and rows == "sample":
        rows = sample_rows(M, x=inp.x)
    return compare(op, inp, out, rows=rows), inp, out

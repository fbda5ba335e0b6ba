"""GPU-vs-oracle comparison with the stated tolerances.

Both sides read the same seeded host tensors (``rmsnorm_norm_fwd_gb300.inputs``).
The GPU side goes through the Python binding, i.e. the C ABI; the oracle is
the fp64 C implementation in ``oracle/``.

Tolerances (per element unless stated; ulp_T(v) is the spacing of dtype T at
|v| with v first rounded to T, the smallest subnormal spacing at 0):
  y      : |dy| <= ulp_T(rnd_T(y_ref))            (bf16; fp16 also accepts
           2e-3 |y_ref|; fp32: 2e-5 (|xhat gamma| + |beta|))
           + 4 * 2^-24 (|xhat gamma| + |beta|)   (fp32 floor for y = xhat*gamma + beta)
           + |gamma_j| (rstd |d_mean| + |xhat_j| e_r)  (the measured error of the
           kernel's own fp32 mean and rstd, carried into y; matters only where
           y = xhat gamma + beta cancels; e_r and d_mean as for dx below)
  rstd   : |d| <= 1e-5 * rstd_ref
  mean   : |d| <= 1e-5 * (|mean_ref| + sqrt(var_ref))
  dx     : |d| <= 2 ulp_T(rnd_T(dx_ref))
                  + u rstd (8 (|g_j| + |c1| + |xhat_j c2|) + K_N (|xhat_j| S2 + S1))
                  + e_r (|dx_j| + 2 rstd |xhat_j c2|) + rstd^2 |d_mean| (|c2| + |xhat_j c1|)
           with u = 2^-24, S2 = (1/N) sum_k |g_k xhat_k|, S1 = (1/N) sum_k |g_k| (LN; 0
           for RMS), K_N = ceil(N/256) + 128.  The second line is the fp32
           arithmetic of dx = rstd (g - c1 - xhat c2): the final operations (8u on
           each term) and the two row sums c2 and c1, each a serial fp32 sum of at
           most ceil(N/256) + 64 terms per thread combined by at most 64 more
           additions, so its error is below K_N u times the sum of magnitudes.  The
           third line carries the measured error of the saved statistics the
           backward reads (e_r = |rstd_gpu - rstd_ref| / rstd_ref, d_mean =
           mean_gpu - mean_ref): rstd enters dx directly, through xhat and through
           c2; the mean through xhat.  For bf16/fp16 the 2-ulp term dominates.
  dgamma, dbeta : ||d||_2 <= 1e-3 ||ref||_2
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
from rmsnorm_norm_fwd_gb300.inputs import DTYPES, make_inputs

MANT = {"bf16": 7, "fp16": 10, "fp32": 23}
EMIN = {"bf16": -126, "fp16": -14, "fp32": -126}
U32 = 2.0 ** -24


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


def y_bound(y_ref, xg_abs, beta_abs, dtype, gam_abs, xhat_abs, rstd, e_r, d_mean):
    floor = 4 * U32 * (xg_abs + beta_abs) + \
        gam_abs[None, :] * (rstd[:, None] * np.abs(d_mean)[:, None] + xhat_abs * e_r[:, None])
    if dtype == "fp32":
        return 2e-5 * (xg_abs + beta_abs) + 1e-30 + floor
    b = ulp(y_ref, dtype)
    if dtype == "fp16":
        b = np.maximum(b, 2e-3 * np.abs(y_ref))
    return b + floor


def dx_bound(dx_ref, rstd, g, c1, xhat, c2, s1, s2, e_r, d_mean, dtype):
    n = dx_ref.shape[1]
    k_n = -(-n // 256) + 128
    r = rstd[:, None]
    terms = np.abs(g) + np.abs(c1)[:, None] + np.abs(xhat * c2[:, None])
    arith = U32 * r * (8 * terms + k_n * (np.abs(xhat) * s2[:, None] + s1[:, None]))
    stats = e_r[:, None] * (np.abs(dx_ref) + 2 * r * np.abs(xhat * c2[:, None])) + \
        r * r * np.abs(d_mean)[:, None] * (np.abs(c2)[:, None] + np.abs(xhat * c1[:, None]))
    return 2 * ulp(dx_ref, dtype) + arith + stats


@dataclass
class Report:
    ok: bool = True
    msgs: list = field(default_factory=list)
    stats: dict = field(default_factory=dict)

    def check_elem(self, name, got, ref, bound):
        err = np.abs(got.astype(np.float64) - ref)
        bad = ~(err <= bound)  # NaN counts as bad
        self.stats[name] = {"max_err": float(np.nanmax(err)) if err.size else 0.0,
                            "max_err_over_bound": float(np.nanmax(err / bound)) if err.size else 0.0,
                            "n_bad": int(bad.sum()), "n": int(err.size)}
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

    def assert_ok(self):
        assert self.ok, "; ".join(self.msgs)


def _np(t):
    return t.detach().to("cpu").double().numpy()


def gpu_run(op, inp, device="cuda", x_dev=None, dy_dev=None):
    """Forward and backward on the GPU through the binding; returns host tensors."""
    import rmsnorm_norm_fwd_gb300 as g
    x = inp.x.to(device) if x_dev is None else x_dev
    dy = inp.dy.to(device) if dy_dev is None else dy_dev
    gamma = inp.gamma.to(device)
    beta = inp.beta.to(device)
    out = {}
    if op == "rms":
        y, rstd = g.rmsnorm_fwd(x, gamma, inp.eps)
        dx, dgam = g.rmsnorm_bwd(dy, x, gamma, rstd)
        out.update(y=y, rstd=rstd, dx=dx, dgamma=dgam)
    else:
        y, mean, rstd = g.layernorm_fwd(x, gamma, beta, inp.eps)
        dx, dgam, dbet = g.layernorm_bwd(dy, x, gamma, mean, rstd)
        out.update(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dgam, dbeta=dbet)
    torch.cuda.synchronize()
    return out


def compare(op, inp, out, rows=None) -> Report:
    """Compare GPU outputs against the oracle.  rows=None: every row; else the
    listed rows for y/stats/dx (dgamma/dbeta always over all rows)."""
    rep = Report()
    dt = inp.dtype
    x = inp.x if rows is None else inp.x[rows]
    dy = inp.dy if rows is None else inp.dy[rows]
    sel = (lambda t: t) if rows is None else (lambda t: t[rows])
    gam = _np(inp.gamma)
    bet = _np(inp.beta) if op == "ln" else np.zeros_like(gam)
    if op == "rms":
        y_ref, rstd_ref = oracle.rmsnorm_fwd(x, inp.gamma, inp.eps)
        mean_ref = np.zeros_like(rstd_ref)
        dx_ref, _ = oracle.rmsnorm_bwd(dy, x, inp.gamma, inp.eps, want_dgamma=False)
        _, dg_ref = oracle.rmsnorm_bwd(inp.dy, inp.x, inp.gamma, inp.eps, want_dx=False)
        db_ref = None
    else:
        y_ref, mean_ref, rstd_ref = oracle.layernorm_fwd(x, inp.gamma, inp.beta, inp.eps)
        dx_ref, _, _ = oracle.layernorm_bwd(dy, x, inp.gamma, inp.eps, want_dparams=False)
        _, dg_ref, db_ref = oracle.layernorm_bwd(inp.dy, inp.x, inp.gamma, inp.eps, want_dx=False)
    xn = _np(x)
    xhat = (xn - mean_ref[:, None]) * rstd_ref[:, None]
    zeros = np.zeros(xn.shape[0])
    e_r = np.abs(_np(sel(out["rstd"])) - rstd_ref) / rstd_ref
    d_mean = _np(sel(out["mean"])) - mean_ref if op == "ln" else zeros
    rep.check_elem("y", _np(sel(out["y"])), y_ref,
                   y_bound(y_ref, np.abs(xhat * gam), np.abs(bet), dt, np.abs(gam), np.abs(xhat),
                           rstd_ref, e_r, d_mean))
    rep.check_elem("rstd", _np(sel(out["rstd"])), rstd_ref, 1e-5 * rstd_ref)
    if op == "ln":
        sd = np.sqrt(np.maximum(1.0 / rstd_ref ** 2 - inp.eps, 0.0))
        rep.check_elem("mean", _np(sel(out["mean"])), mean_ref, 1e-5 * (np.abs(mean_ref) + sd))
    g = _np(dy) * gam
    n = xn.shape[1]
    c1 = g.sum(axis=1) / n if op == "ln" else zeros
    c2 = (g * xhat).sum(axis=1) / n
    s1 = np.abs(g).sum(axis=1) / n if op == "ln" else zeros
    s2 = np.abs(g * xhat).sum(axis=1) / n
    rep.check_elem("dx", _np(sel(out["dx"])), dx_ref,
                   dx_bound(dx_ref, rstd_ref, g, c1, xhat, c2, s1, s2, e_r, d_mean, dt))
    rep.check_l2("dgamma", _np(out["dgamma"]), dg_ref)
    if op == "ln":
        rep.check_l2("dbeta", _np(out["dbeta"]), db_ref)
    return rep


def sample_rows(M: int, k: int = 62, seed: int = 5) -> np.ndarray:
    rng = np.random.default_rng(seed)
    r = set(rng.choice(M, size=min(k, M), replace=False).tolist()) | {0, M - 1}
    return np.array(sorted(r), dtype=np.int64)


def run_case(op, dtype, M, N, dist=None, rows=None, seed=None):
    kw = {} if seed is None else {"seed": seed}
    inp = make_inputs(M, N, dtype=dtype, dist=dist or ("ln" if op == "ln" else "rms"), op=op, **kw)
    out = gpu_run(op, inp)
    return compare(op, inp, out, rows=rows), inp, out

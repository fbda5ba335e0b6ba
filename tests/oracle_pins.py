"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
what the definitions and the mathematics fix:

* hand-worked examples with exact rational answers (``tests/golden``),
* central finite differences of L = sum(dy * y) through the oracle's own
  forward (Richardson-extrapolated, fp64) for dx, dgamma and dbeta,
* closed-form invariants of the normalised row and of the gradients,
* special cases (constant, zero, one-hot rows, N = 1),
* torch.nn.functional.rms_norm / layer_norm with autograd in float64 on the
  CPU -- an independent library, used here only as a cross-check.

They are plain functions (not tests) so that ``test_oracle_mutants`` can run
the same pins against copies of the oracle with a planted mistake.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------- fixtures
def load_worked(name: str) -> dict:
    """Parse a worked-example fixture: 'key: a b ; c d' lines of fractions."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            key, val = key.strip(), val.strip()
            if key == "op":
                out[key] = val
                continue
            rows = [[Fraction(t) for t in r.split()] for r in val.split(";")]
            out[key] = rows
    return out


def _arr(rows) -> np.ndarray:
    a = np.array([[float(v) for v in r] for r in rows], dtype=np.float64)
    return a


def _close(got, want, rtol, atol=0.0, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} out of tolerance; "
                           f"max err {err.max():.3e} (rtol {rtol}, atol {atol})")


def pin_worked_rms():
    w = load_worked("rmsnorm_worked.txt")
    eps = float(w["eps"][0][0])
    x, gamma, dy = _arr(w["x"]), _arr(w["gamma"])[0], _arr(w["dy"])
    y, rstd = oracle.rmsnorm_fwd(x, gamma, eps)
    _close(y, _arr(w["y"]), 1e-14, 1e-15, "rms worked y")
    _close(rstd, _arr(w["rstd"]).ravel(), 1e-14, 0, "rms worked rstd")
    dx, dg = oracle.rmsnorm_bwd(dy, x, gamma, eps)
    _close(dx, _arr(w["dx"]), 1e-13, 1e-15, "rms worked dx")
    _close(dg, _arr(w["dgamma"])[0], 1e-13, 1e-15, "rms worked dgamma")


def pin_worked_ln():
    w = load_worked("layernorm_worked.txt")
    eps = float(w["eps"][0][0])
    x, gamma, beta, dy = _arr(w["x"]), _arr(w["gamma"])[0], _arr(w["beta"])[0], _arr(w["dy"])
    y, mean, rstd = oracle.layernorm_fwd(x, gamma, beta, eps)
    _close(y, _arr(w["y"]), 1e-14, 1e-15, "ln worked y")
    _close(mean, _arr(w["mean"]).ravel(), 1e-14, 0, "ln worked mean")
    _close(rstd, _arr(w["rstd"]).ravel(), 1e-14, 0, "ln worked rstd")
    dx, dg, db = oracle.layernorm_bwd(dy, x, gamma, eps)
    _close(dx, _arr(w["dx"]), 1e-13, 1e-15, "ln worked dx")
    _close(dg, _arr(w["dgamma"])[0], 1e-13, 1e-15, "ln worked dgamma")
    _close(db, _arr(w["dbeta"])[0], 1e-13, 1e-15, "ln worked dbeta")


# --------------------------------------------------------------------------- finite differences
def _loss(op, x, gamma, beta, dy, eps):
    if op == "rms":
        y, _ = oracle.rmsnorm_fwd(x, gamma, eps)
    else:
        y, _, _ = oracle.layernorm_fwd(x, gamma, beta, eps)
    return float(np.sum(dy * y))


def _fd(f, v: np.ndarray, idx, h: float) -> float:
    """Richardson-extrapolated central difference of f along v[idx]."""
    def cd(step):
        a = v.copy()
        b = v.copy()
        a[idx] += step
        b[idx] -= step
        return (f(a) - f(b)) / (2.0 * step)
    d1, d2 = cd(h), cd(h / 2)
    return (4.0 * d2 - d1) / 3.0


def fd_case(op: str, M: int, N: int, seed: int, eps: float):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.3, 1.5, (M, N))
    gamma = 1.0 + 0.3 * rng.normal(size=N)
    beta = 0.2 * rng.normal(size=N)
    dy = rng.normal(size=(M, N))
    if op == "rms":
        dx, dg = oracle.rmsnorm_bwd(dy, x, gamma, eps)
        db = None
    else:
        dx, dg, db = oracle.layernorm_bwd(dy, x, gamma, eps)
    h = 1e-4
    fdx = np.zeros_like(x)
    for i in range(M):
        for j in range(N):
            fdx[i, j] = _fd(lambda v: _loss(op, v, gamma, beta, dy, eps), x, (i, j), h)
    fdg = np.array([_fd(lambda v: _loss(op, x, v, beta, dy, eps), gamma, (j,), h) for j in range(N)])
    scale = max(1.0, np.abs(fdx).max())
    _close(dx, fdx, 0, 1e-8 * scale, f"{op} FD dx M={M} N={N}")
    _close(dg, fdg, 0, 1e-8 * max(1.0, np.abs(fdg).max()), f"{op} FD dgamma M={M} N={N}")
    if op == "ln":
        fdb = np.array([_fd(lambda v: _loss(op, x, gamma, v, dy, eps), beta, (j,), h) for j in range(N)])
        _close(db, fdb, 0, 1e-8 * max(1.0, np.abs(fdb).max()), f"ln FD dbeta M={M} N={N}")


def pin_finite_differences():
    for op in ("rms", "ln"):
        for (M, N) in ((1, 1), (2, 2), (3, 3), (2, 7), (2, 16)):
            fd_case(op, M, N, seed=M * 100 + N, eps=1e-2 if op == "rms" else 1e-1)


# --------------------------------------------------------------------------- invariants
def pin_forward_invariants():
    rng = np.random.default_rng(7)
    M, N = 6, 37
    x = rng.normal(0.5, 2.0, (M, N))
    ones, zeros = np.ones(N), np.zeros(N)
    # RMS of the normalised row (gamma = 1) is sqrt(ms / (ms + eps)).
    eps = 0.3
    y, rstd = oracle.rmsnorm_fwd(x, ones, eps)
    ms = np.mean(x * x, axis=1)
    _close(np.sqrt(np.mean(y * y, axis=1)), np.sqrt(ms / (ms + eps)), 1e-13, 0, "rms(xhat)")
    # Output scaled by gamma column-wise.
    gam = rng.normal(size=N)
    yg, _ = oracle.rmsnorm_fwd(x, gam, eps)
    _close(yg, y * gam, 1e-14, 1e-15, "rms gamma scaling")
    # Scale invariance: y(c x; c^2 eps) == y(x; eps), bit-exact for c = 2^k.
    y4, r4 = oracle.rmsnorm_fwd(4.0 * x, gam, 16.0 * eps)
    assert np.array_equal(y4, yg), "rms scale invariance (c=4) not bit-exact"
    assert np.array_equal(r4, rstd / 4.0), "rms rstd scaling (c=4) not bit-exact"
    # LayerNorm: xhat has mean 0 and variance var/(var+eps); shift invariance.
    eps = 0.2
    y, mean, rstd = oracle.layernorm_fwd(x, ones, zeros, eps)
    var = np.var(x, axis=1)
    _close(np.mean(y, axis=1), np.zeros(M), 0, 1e-14, "ln mean(xhat)")
    _close(np.var(y, axis=1), var / (var + eps), 1e-13, 0, "ln var(xhat)")
    _close(mean, np.mean(x, axis=1), 1e-14, 1e-15, "ln mean")
    ys, _, _ = oracle.layernorm_fwd(x + 3.0, ones, zeros, eps)
    _close(ys, y, 0, 1e-12, "ln shift invariance")
    bet = rng.normal(size=N)
    yb, _, _ = oracle.layernorm_fwd(x, gam, bet, eps)
    _close(yb, y * gam + bet, 1e-14, 1e-14, "ln affine")
    y4, m4, r4 = oracle.layernorm_fwd(4.0 * x, gam, bet, 16.0 * eps)
    _close(y4, yb, 1e-14, 1e-14, "ln scale invariance")


def pin_backward_invariants():
    rng = np.random.default_rng(11)
    M, N = 5, 29
    x = rng.normal(0.5, 2.0, (M, N))
    gamma = 1.0 + 0.1 * rng.normal(size=N)
    dy = rng.normal(size=(M, N))
    g = dy * gamma
    # LayerNorm: sum_j dx_j = 0; sum_j xhat_j dx_j = rstd^3 eps sum_j xhat_j g_j.
    eps = 0.25
    dx, dg, db = oracle.layernorm_bwd(dy, x, gamma, eps)
    _, mean, rstd = oracle.layernorm_fwd(x, gamma, np.zeros(N), eps)
    xhat = (x - mean[:, None]) * rstd[:, None]
    _close(dx.sum(axis=1), np.zeros(M), 0, 1e-13 * np.abs(dx).max(), "ln sum dx")
    _close((xhat * dx).sum(axis=1), rstd ** 3 * eps * (xhat * g).sum(axis=1), 1e-11, 1e-14,
           "ln xhat.dx")
    _close(db, dy.sum(axis=0), 1e-14, 1e-14, "ln dbeta = column sum of dy")
    _close(dg, (dy * xhat).sum(axis=0), 1e-13, 1e-14, "ln dgamma")
    # dy = 1: dbeta = M, and sum_j dgamma_j = sum_ij xhat_ij = 0.
    ones = np.ones((M, N))
    _, dg1, db1 = oracle.layernorm_bwd(ones, x, gamma, eps)
    _close(db1, np.full(N, float(M)), 0, 0, "ln dbeta(dy=1)")
    assert abs(dg1.sum()) < 1e-12 * np.abs(dg1).sum() + 1e-13, "ln sum dgamma(dy=1) != 0"
    # RMSNorm: sum_j x_j dx_j = rstd^3 eps sum_j x_j g_j; zero when eps = 0.
    eps = 0.4
    dx, dg = oracle.rmsnorm_bwd(dy, x, gamma, eps)
    _, rstd = oracle.rmsnorm_fwd(x, gamma, eps)
    _close((x * dx).sum(axis=1), rstd ** 3 * eps * (x * g).sum(axis=1), 1e-11, 1e-14, "rms x.dx")
    _close(dg, (dy * x * rstd[:, None]).sum(axis=0), 1e-13, 1e-14, "rms dgamma")
    dx0, _ = oracle.rmsnorm_bwd(dy, x, gamma, 0.0)
    _close((x * dx0).sum(axis=1), np.zeros(M), 0, 1e-12 * np.abs(x * dx0).sum(), "rms x.dx (eps=0)")


def pin_special_cases():
    N = 8
    gamma = np.linspace(0.5, 2.0, N)
    beta = np.linspace(-1.0, 1.0, N)
    eps = 1e-5
    # Zero row: rstd = 1/sqrt(eps), y = 0 (RMS) or beta (LN).
    z = np.zeros((1, N))
    y, r = oracle.rmsnorm_fwd(z, gamma, eps)
    assert np.all(y == 0) and abs(r[0] - 1 / np.sqrt(eps)) < 1e-12 * r[0]
    # Constant row for LN: var = 0, xhat = 0, y = beta, dgamma = 0, and since
    # d xhat_j / d x_k = rstd (delta_jk - 1/N) there, dx = (g - mean(g)) / sqrt(eps).
    c = np.full((2, N), 3.25)
    y, m, r = oracle.layernorm_fwd(c, gamma, beta, eps)
    _close(y, np.tile(beta, (2, 1)), 0, 1e-15, "ln constant row")
    assert np.all(m == 3.25)
    dx, dg, db = oracle.layernorm_bwd(np.ones((2, N)), c, gamma, eps)
    want = np.tile((gamma - gamma.mean()) / np.sqrt(eps), (2, 1))
    _close(dx, want, 1e-12, 1e-12, "ln constant row dx")
    _close(dg, np.zeros(N), 0, 1e-15, "ln constant row dgamma")
    # One-hot row for RMS: x = a e_k; ms = a^2/N.
    a, k = 3.0, 5
    oh = np.zeros((1, N))
    oh[0, k] = a
    y, r = oracle.rmsnorm_fwd(oh, gamma, eps)
    want = np.zeros(N)
    want[k] = a / np.sqrt(a * a / N + eps) * gamma[k]
    _close(y[0], want, 1e-14, 0, "rms one-hot")
    # N = 1: RMS y = x gamma / sqrt(x^2 + eps); LN y = beta, dx = 0.
    x1 = np.array([[2.0], [-0.5]])
    y, _ = oracle.rmsnorm_fwd(x1, np.array([1.5]), eps)
    _close(y[:, 0], x1[:, 0] * 1.5 / np.sqrt(x1[:, 0] ** 2 + eps), 1e-14, 0, "rms N=1")
    y, _, _ = oracle.layernorm_fwd(x1, np.array([1.5]), np.array([0.25]), eps)
    _close(y[:, 0], np.array([0.25, 0.25]), 0, 0, "ln N=1")
    dx, dg, db = oracle.layernorm_bwd(np.array([[1.0], [2.0]]), x1, np.array([1.5]), eps)
    _close(dx, np.zeros((2, 1)), 0, 0, "ln N=1 dx")
    _close(db, np.array([3.0]), 0, 0, "ln N=1 dbeta")


# --------------------------------------------------------------------------- library cross-check
def pin_torch_fp64():
    gen = torch.Generator().manual_seed(3)
    for (M, N) in ((1, 1), (3, 5), (4, 64), (2, 257), (7, 1000)):
        x = torch.randn(M, N, generator=gen, dtype=torch.float64) * 1.7 + 0.4
        gamma = 1 + 0.2 * torch.randn(N, generator=gen, dtype=torch.float64)
        beta = 0.1 * torch.randn(N, generator=gen, dtype=torch.float64)
        dy = torch.randn(M, N, generator=gen, dtype=torch.float64)
        for op in ("rms", "ln"):
            eps = 1e-6 if op == "rms" else 1e-5
            xt = x.clone().requires_grad_(True)
            gt = gamma.clone().requires_grad_(True)
            bt = beta.clone().requires_grad_(True)
            if op == "rms":
                yt = torch.nn.functional.rms_norm(xt, (N,), gt, eps)
            else:
                yt = torch.nn.functional.layer_norm(xt, (N,), gt, bt, eps)
            yt.backward(dy)
            if op == "rms":
                y, _ = oracle.rmsnorm_fwd(x.numpy(), gamma.numpy(), eps)
                dx, dg = oracle.rmsnorm_bwd(dy.numpy(), x.numpy(), gamma.numpy(), eps)
            else:
                y, _, _ = oracle.layernorm_fwd(x.numpy(), gamma.numpy(), beta.numpy(), eps)
                dx, dg, db = oracle.layernorm_bwd(dy.numpy(), x.numpy(), gamma.numpy(), eps)
                _close(db, bt.grad.numpy(), 1e-12, 1e-12, f"torch dbeta {M}x{N}")
            _close(y, yt.detach().numpy(), 1e-12, 1e-13, f"torch {op} y {M}x{N}")
            # dx = rstd * (g - ...) cancels to ~eps-sized values when N = 1, so the
            # absolute floor scales with the size of the terms, rstd * |g|.
            rs = 1.0 / np.sqrt(np.mean(x.numpy() ** 2, axis=1).min() + eps)
            sdx = max(float(np.abs(dx).max()), rs * float(np.abs(dy.numpy() * gamma.numpy()).max()))
            _close(dx, xt.grad.numpy(), 0, 1e-11 * sdx, f"torch {op} dx {M}x{N}")
            _close(dg, gt.grad.numpy(), 1e-11, 1e-12, f"torch {op} dgamma {M}x{N}")


# --------------------------------------------------------------------------- residual add + norm
_DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
_PREC = {"bf16": (8, -126), "fp16": (11, -14), "fp32": (24, -126)}  # significand bits, min exponent


def round_exact(q: Fraction, dtype: str) -> Fraction:
    """q rounded to the nearest value of dtype, ties to even, in exact
    rational arithmetic (normal and subnormal range; no overflow)."""
    if q == 0:
        return Fraction(0)
    p, emin = _PREC[dtype]
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum = Fraction(2) ** (max(e, emin) - (p - 1))
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return (fl * quantum) * (1 if q > 0 else -1)


def pin_residual_rounding():
    """h = x + r rounded once to the storage type, against exact rational
    sums rounded by hand: random pairs with exponents up to 40 apart, and sums
    that fall exactly on a rounding midpoint (ties go to the even value)."""
    rng = np.random.default_rng(17)
    for dtype, t in _DT.items():
        p, _ = _PREC[dtype]
        xs = rng.normal(size=300) * np.exp2(rng.integers(-10, 10, 300))
        rs = rng.normal(size=300) * np.exp2(rng.integers(-40, 10, 300))
        x = torch.tensor(xs).to(t)
        r = torch.tensor(rs).to(t)
        one, half = 1.0, 2.0 ** -p  # half an ulp of 1
        x = torch.cat([x, torch.tensor([one, one + 2 * half, -one, 3.0]).to(t)])
        r = torch.cat([r, torch.tensor([half, half, -half, 6 * half]).to(t)])
        h = oracle.residual_add(x, r, dtype)
        assert h.dtype == t
        for xi, ri, hi in zip(x.double().tolist(), r.double().tolist(), h.double().tolist()):
            want = round_exact(Fraction(xi) + Fraction(ri), dtype)
            assert Fraction(hi) == want, f"{dtype}: {xi!r} + {ri!r} -> {hi!r}, want {float(want)!r}"
        # the midpoints: 1 + half -> 1 (even); (1 + 2 half) + half -> 1 + 4 half
        assert h[-4].item() == 1.0 and h[-3].item() == 1.0 + 4 * half and h[-2].item() == -1.0


def pin_residual_worked():
    w = load_worked("residual_worked.txt")
    eps = float(w["eps"][0][0])
    x, r, gamma = _arr(w["x"]), _arr(w["r"]), _arr(w["gamma"])[0]
    dy, dres = _arr(w["dy"]), _arr(w["dres"])
    for dtype in ("bf16", "fp16", "fp32"):
        h = oracle.residual_add(x, r, dtype)
        _close(h.double().numpy(), _arr(w["h"]), 0, 0, f"residual worked h {dtype}")
        y, rstd = oracle.rmsnorm_fwd(h, gamma, eps)
        _close(y, _arr(w["y"]), 1e-14, 1e-15, "residual worked y")
        _close(rstd, _arr(w["rstd"]).ravel(), 1e-14, 0, "residual worked rstd")
        dx, dg = oracle.rmsnorm_bwd(dy, h, gamma, eps, dres=dres)
        _close(dx, _arr(w["dx"]), 1e-13, 1e-15, "residual worked dx")
        _close(dg, _arr(w["dgamma"])[0], 1e-13, 1e-15, "residual worked dgamma")


def pin_residual_finite_differences():
    """With the exact sum (no rounding), the gradient of
    L = sum dy * norm(x + r) + sum dres * (x + r) with respect to x and to r
    both equal the oracle's dx with dres added."""
    for op in ("rms", "ln"):
        for (M, N) in ((1, 3), (2, 5), (2, 16)):
            rng = np.random.default_rng(M * 31 + N)
            x = rng.normal(0.2, 1.3, (M, N))
            r = rng.normal(-0.1, 0.7, (M, N))
            gamma = 1.0 + 0.3 * rng.normal(size=N)
            beta = 0.2 * rng.normal(size=N)
            dy = rng.normal(size=(M, N))
            dres = rng.normal(size=(M, N))
            eps = 1e-2

            def loss(xv, rv):
                h = oracle.residual_add(xv, rv, None)
                return _loss(op, h, gamma, beta, dy, eps) + float(np.sum(dres * h))

            h = oracle.residual_add(x, r, None)
            if op == "rms":
                dx, _ = oracle.rmsnorm_bwd(dy, h, gamma, eps, dres=dres)
            else:
                dx, _, _ = oracle.layernorm_bwd(dy, h, gamma, eps, dres=dres)
            for which in ("x", "r"):
                fd = np.zeros_like(x)
                for i in range(M):
                    for j in range(N):
                        if which == "x":
                            fd[i, j] = _fd(lambda v: loss(v, r), x, (i, j), 1e-4)
                        else:
                            fd[i, j] = _fd(lambda v: loss(x, v), r, (i, j), 1e-4)
                _close(dx, fd, 0, 1e-8 * max(1.0, np.abs(fd).max()), f"{op} residual FD d{which} {M}x{N}")


def pin_residual_special_cases():
    """r = 0 stores h = x and normalises x; dres = 0 leaves dx as the plain
    backward; for LayerNorm, dx - dres sums to zero along each row."""
    rng = np.random.default_rng(23)
    M, N = 4, 24
    x = torch.tensor(rng.normal(size=(M, N))).to(torch.bfloat16)
    gamma = 1.0 + 0.1 * rng.normal(size=N)
    dy = rng.normal(size=(M, N))
    h = oracle.residual_add(x, torch.zeros(M, N, dtype=torch.bfloat16), "bf16")
    assert torch.equal(h, x)
    dx0, _ = oracle.rmsnorm_bwd(dy, h, gamma, 1e-6)
    dxz, _ = oracle.rmsnorm_bwd(dy, h, gamma, 1e-6, dres=np.zeros((M, N)))
    assert np.array_equal(dx0, dxz)
    dres = rng.normal(size=(M, N))
    dxl, _, _ = oracle.layernorm_bwd(dy, h, gamma, 1e-5, dres=dres)
    _close((dxl - dres).sum(axis=1), np.zeros(M), 0, 1e-12, "ln residual: sum (dx - dres) = 0")


ALL_PINS = [pin_worked_rms, pin_worked_ln, pin_finite_differences, pin_forward_invariants,
            pin_backward_invariants, pin_special_cases, pin_torch_fp64, pin_residual_rounding,
            pin_residual_worked, pin_residual_finite_differences, pin_residual_special_cases]

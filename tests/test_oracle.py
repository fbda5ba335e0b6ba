"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()


def test_worked_fixtures_are_exact_by_construction():
    """The hand-worked fixtures satisfy the definitions in exact rational arithmetic.

    This checks the fixtures themselves (not the oracle): every stated mean,
    rstd and y follows from the stated x, gamma, beta and eps with Fractions,
    and rstd^-2 equals the mean square (or variance) plus eps exactly.
    """
    from fractions import Fraction as F
    w = P.load_worked("rmsnorm_worked.txt")
    eps = w["eps"][0][0]
    for xr, yr, (r,) in zip(w["x"], w["y"], w["rstd"]):
        ms = sum(v * v for v in xr) / len(xr)
        assert 1 / (r * r) == ms + eps
        assert [v * r * g for v, g in zip(xr, w["gamma"][0])] == yr
    w = P.load_worked("layernorm_worked.txt")
    eps = w["eps"][0][0]
    for xr, yr, (mu,), (r,) in zip(w["x"], w["y"], w["mean"], w["rstd"]):
        n = len(xr)
        assert sum(xr) / n == mu
        var = sum((v - mu) ** 2 for v in xr) / n
        assert 1 / (r * r) == var + eps
        assert [(v - mu) * r * g + b for v, g, b in zip(xr, w["gamma"][0], w["beta"][0])] == yr
    assert F(0) == sum(w["dx"][0]) == sum(w["dx"][1])  # LayerNorm: each dx row sums to zero


def test_residual_fixture_is_exact_by_construction():
    """The residual fixture: h = x + r exactly; its rows are the worked RMSNorm
    rows (same eps, gamma, dy, so the same y and dgamma); dx is that example's
    dx plus dres."""
    r = P.load_worked("residual_worked.txt")
    w = P.load_worked("rmsnorm_worked.txt")
    assert r["eps"] == w["eps"] and r["gamma"] == w["gamma"] and r["dy"] == w["dy"]
    assert [[a + b for a, b in zip(xr, rr)] for xr, rr in zip(r["x"], r["r"])] == r["h"] == w["x"]
    assert r["y"] == w["y"] and r["rstd"] == w["rstd"] and r["dgamma"] == w["dgamma"]
    assert [[a + b for a, b in zip(dr, sr)] for dr, sr in zip(w["dx"], r["dres"])] == r["dx"]

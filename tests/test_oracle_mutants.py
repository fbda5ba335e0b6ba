"""Plants one plausible mistake at a time in a copy of the oracle's C source and
checks that the pins catch every one of them (CPU only).

The mutants are compiled into temporary libraries and swapped in for the real
one only for the duration of each case; the oracle on disk is never changed.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "norm_oracle.c")

# (name, original text, mutated text): each a mistake a careful reader could make.
MUTANTS = [
    ("unbiased_variance", "        s += d * d;\n    }\n    return s / (double)N;",
     "        s += d * d;\n    }\n    return s / (double)(N > 1 ? N - 1 : 1);"),
    ("rms_eps_dropped", "double r = 1.0 / sqrt(ms + eps);", "double r = 1.0 / sqrt(ms);"),
    ("ln_eps_outside_root", "double r = 1.0 / sqrt(var + eps);", "double r = 1.0 / sqrt(var) + eps;"),
    ("ln_mean_not_subtracted", "yr[j] = ((xr[j] - mu) * r) * gamma[j] + beta[j];",
     "yr[j] = (xr[j] * r) * gamma[j] + beta[j];"),
    ("ln_beta_dropped", "yr[j] = ((xr[j] - mu) * r) * gamma[j] + beta[j];",
     "yr[j] = ((xr[j] - mu) * r) * gamma[j];"),
    ("rms_gamma_wrong_index", "yr[j] = (xr[j] * r) * gamma[j];", "yr[j] = (xr[j] * r) * gamma[N - 1 - j];"),
    ("ln_dx_sign", "(g - mean_g - xhat * mean_gxhat)", "(g + mean_g - xhat * mean_gxhat)"),
    ("rms_dx_term_dropped", ": (g - xhat * mean_gxhat);", ": (g);"),
    ("dx_gamma_dropped", "            double g = dyr[j] * gamma[j];", "            double g = dyr[j];"),
    ("dx_rstd_dropped", "dxr[j] = r * inner;", "dxr[j] = inner;"),
    ("mean_g_not_divided", "        mean_g /= (double)N;\n", "\n"),
    ("dgamma_uses_x", "accg[j - j0] += dyr[j] * xhat;", "accg[j - j0] += dyr[j] * xr[j];"),
    ("dbeta_weighted", "accb[j - j0] += dyr[j];", "accb[j - j0] += dyr[j] * xhat;"),
    ("dgamma_transposed", "double xhat = (xr[j] - mean[ii]) * rstd[ii];",
     "double xhat = (xr[j] - mean[ii]) * rstd[ii > 0 ? ii - 1 : ii];"),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant {name}: anchor text not found exactly once"
    path = tmp_path / f"mut_{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"libmut_{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(path), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    return str(lib)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name, old, new):
    libpath = _build_mutant(tmp_path, name, old, new)
    real = oracle._load()
    mut = ctypes.CDLL(libpath)
    for fn in ("oracle_rmsnorm_fwd", "oracle_layernorm_fwd", "oracle_rmsnorm_bwd",
               "oracle_layernorm_bwd"):
        getattr(mut, fn).argtypes = getattr(real, fn).argtypes
        getattr(mut, fn).restype = getattr(real, fn).restype
    monkeypatch.setattr(oracle, "_lib", mut)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name!r}"


# Mistakes in the residual add + norm part of the oracle (its Python layer),
# planted by wrapping the oracle's functions for the duration of one case.
def _mut_dres_dropped(orig):
    def f(*a, dres=None, **k):
        return orig(*a, **k)
    return f


def _mut_dres_subtracted(orig):
    def f(*a, dres=None, **k):
        return orig(*a, dres=None if dres is None else -oracle._f64(dres), **k)
    return f


def _mut_sum_not_rounded(orig):
    def f(x, r, dtype=None):
        import torch
        return orig(x, r, None) if dtype is None else torch.from_numpy(orig(x, r, None))
    return f


def _mut_residual_not_added(orig):
    def f(x, r, dtype=None):
        return orig(x, 0 * oracle._f64(r), dtype)
    return f


def _mut_round_toward_zero(orig):
    def f(x, r, dtype=None):
        import torch
        h = orig(x, r, dtype)
        if dtype is None:
            return h
        s = torch.from_numpy(oracle._f64(x) + oracle._f64(r))
        # one step toward zero wherever rounding went away from zero
        return torch.where(h.double().abs() > s.abs(), torch.nextafter(h, torch.zeros_like(h)), h)
    return f


RESIDUAL_MUTANTS = [
    ("dres_dropped", ("rmsnorm_bwd", "layernorm_bwd"), _mut_dres_dropped),
    ("dres_subtracted", ("rmsnorm_bwd", "layernorm_bwd"), _mut_dres_subtracted),
    ("sum_not_rounded", ("residual_add",), _mut_sum_not_rounded),
    ("residual_not_added", ("residual_add",), _mut_residual_not_added),
    ("round_toward_zero", ("residual_add",), _mut_round_toward_zero),
]


@pytest.mark.parametrize("name,fns,make", RESIDUAL_MUTANTS, ids=[m[0] for m in RESIDUAL_MUTANTS])
def test_pins_catch_planted_residual_mistake(monkeypatch, name, fns, make):
    for fn in fns:
        monkeypatch.setattr(oracle, fn, make(getattr(oracle, fn)))
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name!r}"

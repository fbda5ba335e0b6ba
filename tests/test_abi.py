"""The C-ABI library: loads, exports every declared symbol, and rejects bad
arguments before touching a device (CPU only; nothing here launches)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")
LIB = os.path.join(ROOT, "rmsnorm_norm_fwd_gb300", "libgbnorm.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from rmsnorm_norm_fwd_gb300 import build
        build.build()
    from rmsnorm_norm_fwd_gb300 import binding
    return binding.lib


def declared_functions():
    names = []
    for h in sorted(os.listdir(HEADER_DIR)):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", text, re.M):
            names.append(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for want in ("rmsnorm_fwd", "rmsnorm_bwd", "layernorm_fwd", "layernorm_bwd",
                 "norm_bwd_workspace_size", "gbnorm_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_exported_symbols_are_c_names():
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in declared_functions():
        assert n in syms, f"{n} not exported with C linkage"


def test_status_strings(lib):
    for s, want in ((0, "ok"), (1, "invalid argument"), (3, "workspace")):
        assert want in lib.gbnorm_status_string(s).decode()
    assert lib.gbnorm_status_string(99) == b"unknown status"


def test_variant_tables(lib):
    from rmsnorm_norm_fwd_gb300 import binding as b
    src = open(os.path.join(ROOT, "rmsnorm_norm_fwd_gb300", "csrc", "api.cu")).read()
    cap = int(re.search(r"constexpr int kMaxVariants = (\d+);", src).group(1))
    for ln in (False, True):
        for d in (0, 1):
            for dt in ("fp32", "fp16", "bf16"):
                names = b.variants(ln, d, dt)
                assert "elem" in names and len(names) == len(set(names)) >= 10
                # the host's per-variant caches are indexed by variant
                assert len(names) <= cap, (ln, d, dt, len(names), cap)
    assert lib.gbnorm_force_variant(0, 0, 2, b"no-such-variant") == 1
    assert lib.gbnorm_force_variant(0, 0, 2, None) == 0
    assert lib.gbnorm_variant_at(0, 0, 2, 10_000) is None


# Fake, never-dereferenced addresses: argument checks run before any device use.
A, B, C, D, E_, F, G, H = (0x10000 * k for k in range(1, 9))
V = ctypes.c_void_p


def test_forward_rejects_bad_arguments(lib):
    bf16 = 2
    f = lib.rmsnorm_fwd
    assert f(V(A), V(B), V(C), V(D), 4, 0, bf16, 1e-6, None) == 1            # N = 0
    assert f(V(A), V(B), V(C), V(D), -1, 8, bf16, 1e-6, None) == 1           # M < 0
    assert f(V(A), V(B), V(C), V(D), 4, 8, 7, 1e-6, None) == 1               # dtype
    assert f(None, V(B), V(C), V(D), 4, 8, bf16, 1e-6, None) == 1            # x null
    assert f(V(A), V(B), V(C), V(D), 4, 8, bf16, float("nan"), None) == 1    # eps
    assert f(V(A), V(B), V(C), V(D), 4, 8, bf16, -1.0, None) == 1            # eps < 0
    assert f(V(A), V(B), V(A + 2), V(D), 4, 8, bf16, 1e-6, None) == 1        # y overlaps x
    assert f(V(A), V(B), V(C), V(C + 4), 4, 8, bf16, 1e-6, None) == 1        # rstd overlaps y
    assert f(V(A), V(B), V(C), V(D), 4, (1 << 24) + 1, bf16, 1e-6, None) == 1  # N too large
    g = lib.layernorm_fwd
    assert g(V(A), V(B), V(F), V(C), V(D), V(D), 4, 8, bf16, 1e-5, None) == 1   # mean == rstd


def test_backward_rejects_bad_arguments(lib):
    bf16 = 2
    f = lib.rmsnorm_bwd
    # dx overlapping x (not the permitted in-place pair dx == dy)
    assert f(V(A), V(B), V(C), V(D), V(B), V(E_), V(F), 1 << 20, 4, 8, bf16, None) == 1
    assert f(V(A), V(B), V(C), None, V(E_), V(G), V(F), 1 << 20, 4, 8, bf16, None) == 1  # rstd
    assert f(V(A), V(B), V(C), V(D), V(E_), V(G), V(F), 1 << 20, 4, 0, bf16, None) == 1  # N
    g = lib.layernorm_bwd
    assert g(V(A), V(B), V(C), None, V(D), V(E_), V(F), V(G), V(H), 1 << 20, 4, 8, bf16, None) == 1
    assert g(V(A), V(B), V(C), V(D), V(D + 8), V(E_), V(F), V(F), V(H), 1 << 20, 4, 8, bf16,
             None) == 1  # dgamma == dbeta


def test_null_parameters_are_accepted(lib):
    """gamma / beta / dgamma / dbeta may be NULL (the constants 1 / 0, or sums
    not produced), at any N: such calls pass the argument checks; without a
    usable device they report CUDA or unsupported, never invalid arguments."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    bf16 = 2
    assert lib.rmsnorm_fwd(V(A), None, V(C), V(D), 4, 8, bf16, 1e-6, None) in (2, 4)
    assert lib.layernorm_fwd(V(A), None, None, V(C), V(D), V(E_), 4, 8, bf16, 1e-5, None) in (2, 4)
    assert lib.rmsnorm_bwd(V(A), V(B), None, V(D), V(E_), None, V(F), 1 << 20, 4, 8, bf16,
                           None) in (2, 4)
    assert lib.layernorm_bwd(V(A), V(B), None, V(C), V(D), V(E_), None, None, V(H), 1 << 20, 4, 8,
                             bf16, None) in (2, 4)
    # no limit on N for the missing rows: nothing is read for them (buffers
    # 2^40 bytes apart, so that the wide rows do not overlap)
    far = [V(k << 40) for k in range(1, 7)]
    assert lib.rmsnorm_fwd(far[0], None, far[1], far[2], 4, (1 << 20) + 8, bf16, 1e-6, None) in (2, 4)
    assert lib.layernorm_fwd(far[0], far[3], None, far[1], far[2], far[4], 4, (1 << 20) + 8, bf16,
                             1e-5, None) in (2, 4)


def test_valid_call_without_device_reports_cuda_or_unsupported(lib):
    # A well-formed call on a machine without a usable sm_103a device must not
    # pretend to succeed.
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    st = lib.rmsnorm_fwd(V(A), V(B), V(C), V(D), 4, 8, 2, 1e-6, None)
    assert st in (2, 4)
    assert lib.norm_bwd_workspace_size(0, 4, 8, 2) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    env = dict(os.environ, GBNORM_LIB=str(tmp_path / "missing.so"), PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", "import rmsnorm_norm_fwd_gb300 as g; g.rmsnorm_fwd"],
                       capture_output=True, text=True, env=env, cwd=ROOT)
    assert r.returncode != 0 and "libgbnorm.so not found" in r.stderr


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "rmsnorm_norm_fwd_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".inc", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "norm_oracle" not in text, fn


def test_dispatch_table_names_compiled_variants(lib):
    """Every variant the dispatch table names exists in the compiled tables of
    every (op, direction, dtype) its row applies to: a misspelt or removed name
    would otherwise be skipped silently and the row's shapes served by the
    next row."""
    from rmsnorm_norm_fwd_gb300 import binding as b
    table = os.path.join(ROOT, "rmsnorm_norm_fwd_gb300", "csrc", "dispatch_table.inc")
    rows = re.findall(r'^\{(-?\d+), (\d+), (-?\d+), (-?\d+), (\d+), "([^"]+)"\}', open(table).read(), re.M)
    assert len(rows) > 50
    names = {0: "fp32", 1: "fp16", 2: "bf16"}
    for ln, d, dt, m_max, nv, variant in rows:
        assert int(m_max) == -1 or int(m_max) > 0
        for is_ln in ((0, 1) if ln == "-1" else (int(ln),)):
            for code in ((0, 1, 2) if dt == "-1" else (int(dt),)):
                assert variant in b.variants(bool(is_ln), int(d), names[code]), \
                    (variant, is_ln, d, names[code])
        assert int(nv) > 0


def test_general_form_rejects_bad_arguments(lib):
    """norm_fwd_ex / norm_bwd_ex argument checks (before any device use)."""
    bf16, f32 = 2, 0
    I64 = ctypes.c_int64
    lib.norm_fwd_ex.argtypes = [ctypes.c_int, I64, I64, ctypes.c_float, V, I64, ctypes.c_int, V, I64, V, I64, V,
                                V, ctypes.c_int, V, I64, ctypes.c_int, V, V, V]
    f = lib.norm_fwd_ex
    far = [V(k << 40) for k in range(1, 9)]
    M, N = 4, 64
    ok = dict(x=far[0], ldx=N, r=None, ldr=N, h=None, ldh=N, y=far[1], ldy=N)

    def fwd(**kw):
        a = {**ok, **kw}
        return f(0, M, N, 1e-6, a["x"], a["ldx"], bf16, a["r"], a["ldr"], a["h"], a["ldh"], far[2], None, f32,
                 a["y"], a["ldy"], bf16, None, far[3], None)
    assert fwd(h=far[4]) == 1                   # h without a residual
    assert fwd(ldx=N - 1) == 1                  # row stride below N
    assert fwd(ldy=N - 8) == 1
    assert fwd(y=V((1 << 40) + 64)) == 1        # y overlaps x (not the same rows)
    assert fwd(r=far[4], h=V((5 << 40) + 2)) == 1  # h overlaps the residual, not exactly
    assert f(0, M, N, 1e-6, far[0], N, 5, None, N, None, N, None, None, f32, far[1], N, bf16, None, None,
             None) == 1                          # x dtype
    assert f(0, M, N, float("nan"), far[0], N, bf16, None, N, None, N, None, None, f32, far[1], N, bf16, None,
             None, None) == 1                    # eps
    lib.norm_bwd_ex.argtypes = [ctypes.c_int, I64, I64, V, I64, ctypes.c_int, V, I64, ctypes.c_int, V, I64, V,
                                ctypes.c_int, V, V, V, I64, V, V, V, ctypes.c_size_t, V]
    b = lib.norm_bwd_ex
    assert b(0, M, N, far[0], N, bf16, far[1], N, bf16, None, N, None, bf16, None, far[2], far[1], N, None, None,
             far[3], 1 << 20, None) == 1         # dx over x
    assert b(0, M, N, far[0], N, bf16, far[1], N, bf16, None, N, None, bf16, None, None, far[4], N, None, None,
             far[3], 1 << 20, None) == 1         # rstd missing
    assert b(0, M, N, far[0], N - 1, bf16, far[1], N, bf16, None, N, None, bf16, None, far[2], far[4], N, None,
             None, far[3], 1 << 20, None) == 1   # dy row stride below N

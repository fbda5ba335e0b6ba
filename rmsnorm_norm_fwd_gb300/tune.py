"""Measures every kernel variant on the workload shapes and writes the
measured rows of csrc/dispatch_table.inc.

    python -m rmsnorm_norm_fwd_gb300.tune --out sweep.json        # on a GB300
    python -m rmsnorm_norm_fwd_gb300.tune --emit sweep.json       # rewrites the table

Each (op, direction, dtype, N, M) is timed for every variant that can serve
it (forced through gbnorm_force_variant), with L2 flushed before every timed
call (1 GiB write, then 512 MiB read), CUDA events on the launching stream,
median of --reps calls.  The table is keyed on the row count too: shapes with
M <= SMALL_M are measured separately and written as rows that apply only to
calls with at most SMALL_M rows, ahead of the rows for any M.  Effective
bandwidth uses the algorithmic bytes only (b = element size):
    RMS fwd 2MNb + Nb + 4M     LN fwd 2MNb + 2Nb + 8M
    RMS bwd 3MNb + Nb + 4M + 4N   LN bwd 3MNb + Nb + 8M + 8N
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import sys

DTYPE_CODE = {"fp32": 0, "fp16": 1, "bf16": 2}
ELEM = {"fp32": 4, "fp16": 2, "bf16": 2}

# Calls with at most this many rows have their own measured rows.
SMALL_M = 1024

# (op, dtype, M, N) of the workloads, and the small-M bucket of the short and
# LLM-shaped rows.
SHAPES = (
    [(op, "bf16", SMALL_M, n) for op in ("rms", "ln") for n in (256, 512, 1024, 2048, 4096, 8192)]
    + [("rms", "bf16", 65536, n) for n in (256, 384, 512, 768, 1024, 2048)]
    + [("ln", "bf16", 16384, n) for n in (4096, 8192)]
    + [(op, "bf16", 2048, n) for op in ("rms", "ln") for n in (16384, 32768, 65536, 131072)]
    + [(op, dt, 16384, n) for op in ("rms", "ln") for dt in ("bf16", "fp16", "fp32")
       for n in (4096, 5120, 8192)]
)


def alg_bytes(op, direction, M, N, b):
    if direction == 0:
        return 2 * M * N * b + (2 if op == "ln" else 1) * N * b + (8 if op == "ln" else 4) * M
    return 3 * M * N * b + N * b + (8 if op == "ln" else 4) * M + (8 if op == "ln" else 4) * N


def sweep(reps: int, only=None, dirs=(0, 1)):
    import torch

    import rmsnorm_norm_fwd_gb300 as g
    dt_t = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}
    dev = torch.device("cuda")
    # L2 flush before each timed call: a 1 GiB write, then a 512 MiB read so
    # that the lines left in L2 are clean (no write-back inside the timing).
    scrub = torch.empty(1 << 30, device=dev, dtype=torch.uint8)
    clean = torch.ones(128 << 20, device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream()
    out = []
    for op, dt, M, N in SHAPES:
        if only and not re.search(only, f"{op}-{dt}-{M}x{N}"):
            continue
        ln = op == "ln"
        t = dt_t[dt]
        x = torch.randn(M, N, device=dev, dtype=torch.float32).to(t)
        dy = torch.randn(M, N, device=dev, dtype=torch.float32).to(t)
        gam = (1 + 0.1 * torch.randn(N, device=dev)).to(t)
        bet = (0.1 * torch.randn(N, device=dev)).to(t)
        y = torch.empty_like(x)
        dx = torch.empty_like(x)
        mean = torch.empty(M, device=dev)
        rstd = torch.empty(M, device=dev)
        dg = torch.empty(N, device=dev)
        db = torch.empty(N, device=dev)
        if ln:
            g.layernorm_fwd(x, gam, bet, 1e-5, y=y, mean=mean, rstd=rstd)
        else:
            g.rmsnorm_fwd(x, gam, 1e-6, y=y, rstd=rstd)
        for direction in dirs:
            default = g.variant_name(ln, direction, M, N, dt)
            for v in g.variants(ln, direction, dt):
                if v == "elem":
                    continue
                g.force_variant(ln, direction, dt, v)
                try:
                    if g.variant_name(ln, direction, M, N, dt) != v:
                        continue
                    ws = None
                    if direction == 1:
                        ws = torch.empty(g.norm_bwd_workspace_size(ln, M, N, t), device=dev,
                                         dtype=torch.uint8)

                    def call():
                        if direction == 0:
                            if ln:
                                g.layernorm_fwd(x, gam, bet, 1e-5, y=y, mean=mean, rstd=rstd)
                            else:
                                g.rmsnorm_fwd(x, gam, 1e-6, y=y, rstd=rstd)
                        elif ln:
                            g.layernorm_bwd(dy, x, gam, mean, rstd, dx=dx, dgamma=dg, dbeta=db, workspace=ws)
                        else:
                            g.rmsnorm_bwd(dy, x, gam, rstd, dx=dx, dgamma=dg, workspace=ws)

                    call()
                    times = []
                    for _ in range(reps):
                        scrub.zero_()
                        clean.amax()
                        a = torch.cuda.Event(enable_timing=True)
                        b = torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        call()
                        b.record(stream)
                        b.synchronize()
                        times.append(a.elapsed_time(b))
                    ms = statistics.median(times)
                    gbs = alg_bytes(op, direction, M, N, ELEM[dt]) / (ms * 1e-3) / 1e9
                    out.append({"op": op, "dir": direction, "dtype": dt, "M": M, "N": N, "variant": v,
                                "ms": ms, "gbs": gbs, "default": v == default})
                    print(f"{op} {'fwd' if direction == 0 else 'bwd'} {dt} {M}x{N} {v:>16s} "
                          f"{ms * 1e3:8.1f} us {gbs:8.1f} GB/s{'  (default)' if v == default else ''}",
                          flush=True)
                finally:
                    g.force_variant(ln, direction, dt, None)
        del x, dy, y, dx
        torch.cuda.empty_cache()
    if g.read_fault(reset=True):
        raise RuntimeError("a kernel's bounded wait timed out during the sweep")
    return out


ROW_RE = re.compile(r'^\{(\d+), (\d+), (\d+), (-?\d+), (\d+), "[^"]+"\},.*$')


def m_bucket(M: int) -> int:
    """m_max of the table row a measurement at M rows belongs to (-1: any M)."""
    return SMALL_M if M <= SMALL_M else -1


# A measured row keeps its variant unless another one measures faster by
# more than this fraction (CUDA event timestamps advance in steps of about
# 2 us, so short calls tie often).
KEEP_MARGIN = 0.01


def emit(results, table_path):
    """Merge sweep results into the measured block of the dispatch table: a
    (op, direction, dtype, M bucket, N) the sweep measured gets its fastest
    variant (the current one on a near tie, see KEEP_MARGIN); the other
    measured rows stay as they are."""
    best, seen = {}, {}
    for r in results:
        key = (r["op"], r["dir"], r["dtype"], m_bucket(r["M"]), r["N"])
        seen.setdefault(key, {})[r["variant"]] = r
        if key not in best or r["gbs"] > best[key]["gbs"]:
            best[key] = r
    text = open(table_path).read()
    start = text.index("// ---- measured rows (tune.py) ----")
    end = text.index("// ---- forward defaults")
    rows = {}
    current = {}
    for line in text[start:end].splitlines()[1:]:
        m = ROW_RE.match(line)
        if m:
            k = tuple(int(v) for v in m.groups())
            rows[k] = line
            current[k] = re.search(r'"([^"]+)"', line).group(1)
    for (op, d, dt, mb, n), r in list(best.items()):
        k = (1 if op == "ln" else 0, d, DTYPE_CODE[dt], mb, n * ELEM[dt] // 16)
        cur = seen[(op, d, dt, mb, n)].get(current.get(k))
        if cur is not None and cur["gbs"] >= r["gbs"] * (1 - KEEP_MARGIN):
            best[(op, d, dt, mb, n)] = cur
    for (op, d, dt, mb, n), r in best.items():
        key = (1 if op == "ln" else 0, d, DTYPE_CODE[dt], mb, n * ELEM[dt] // 16)
        rows[key] = (f'{{{key[0]}, {d}, {key[2]}, {key[3]}, {key[4]}, "{r["variant"]}"}},'
                     f'  // {op} {"fwd" if d == 0 else "bwd"} {dt} M={r["M"]} N={n}: {r["gbs"]:.0f} GB/s')
    # by row length; for one row length the small-M row first (the first
    # matching row wins)
    order = sorted(rows, key=lambda k: (-k[0], k[1], -k[2], k[4], k[3] < 0, k[3]))
    block = "// ---- measured rows (tune.py) ----\n" + "\n".join(rows[k] for k in order) + "\n"
    open(table_path, "w").write(text[:start] + block + text[end:])
    return [rows[k] for k in order]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--out", help="write sweep results (JSON) here")
    ap.add_argument("--emit", help="read sweep results (JSON) and rewrite the dispatch table")
    ap.add_argument("--reps", type=int, default=7)
    ap.add_argument("--only", help="regex over 'op-dtype-MxN' to restrict the sweep")
    ap.add_argument("--dir", choices=("fwd", "bwd", "both"), default="both", help="directions to sweep")
    a = ap.parse_args(argv)
    here = os.path.dirname(os.path.abspath(__file__))
    if a.emit:
        with open(a.emit) as f:
            rows = emit(json.load(f), os.path.join(here, "csrc", "dispatch_table.inc"))
        print("\n".join(rows))
        return 0
    res = sweep(a.reps, a.only, {"fwd": (0,), "bwd": (1,), "both": (0, 1)}[a.dir])
    if a.out:
        with open(a.out, "w") as f:
            json.dump(res, f)
    return 0


if __name__ == "__main__":
    sys.exit(main())

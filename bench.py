"""Benchmark: fused RMSNorm forward + backward, effective HBM GB/s on GB300.

One step = the whole hot path (forward, backward row kernel, dgamma column
reduce) over the big-M small-N sweep: RMSNorm, M = 65536 rows,
N in {256, 384, 512, 768, 1024, 2048}, bf16 tensors, eps = 1e-6,
x, dy ~ N(0,1), gamma = 1 + 0.1 N(0,1) (seeded synthetic data).

value = algorithmic bytes of every timed call / summed CUDA-event time of
those calls.  Algorithmic bytes per call (b = 2 for bf16):
    forward  : 2 M N b + N b + 4 M          (x, y, gamma, rstd)
    backward : 3 M N b + N b + 4 M + 4 N    (dy, x, dx, gamma, rstd, dgamma)
Workspace traffic counts as time, never as bytes.  L2 is flushed (a 1 GiB
write, then a 512 MiB read so the lines left are clean; outside the events)
before every timed call.

The JSON line's "families" object adds every other workload of the path,
timed per shape and direction in the same run (median of 5 calls, L2 flushed
before each): RMSNorm 1024x1024; LayerNorm 16384 x {4096, 8192}; RMSNorm and
LayerNorm 2048 x {16K, 32K, 64K, 128K}; RMSNorm and LayerNorm 16384 x {4096,
5120, 8192} in bf16, fp16 and fp32 with the accumulation-stress inputs; the
sweep above in the same form; and ("general_form") the strided, mixed-type
and residual-add calls of norm_fwd_ex / norm_bwd_ex at 16384 x 8192.  For each family the largest row length is
held to the targets: forward >= 0.85 and backward >= 0.75 of the measured
copy peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs the same per-GPU workload (weak
scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rmsnorm_norm_fwd_gb300.inputs import make_inputs  # noqa: E402

M = 65536
NS = (256, 384, 512, 768, 1024, 2048)
EPS = 1e-6
B = 2  # bf16
METRIC = "norm fwd/bwd effective HBM GB/s and % of GB300 peak, per (M,N,dtype)"
WORKLOAD = ("RMSNorm fwd+bwd sweep, M=65536 rows, N in {256,384,512,768,1024,2048}, "
            "bf16 tensors, fp32 rstd and dgamma, eps=1e-6")
# Before every timed call: a 1 GiB write (flushes the 129 MB L2 and keeps the
# GPU busy long enough that the host has queued the timed call before the GPU
# reaches its start event), then a 512 MiB read, so that L2 holds clean lines
# of an unrelated buffer instead of dirty ones whose write-back would land in
# the timed call.
L2_FLUSH_BYTES = 1 << 30
L2_CLEAN_BYTES = 512 << 20

# Measured DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the
# roofline kernel, from the ncu capture summarised under profiles/, valid only
# while the code that kernel is compiled and launched from (ROOFLINE_SOURCES:
# its kernel file, the shared device helpers and argument blocks, and the host
# code that dispatches it and sizes its grid and ring) hashes to the digest
# recorded with it.
# api.cu counts up to its argument-check section: the dispatch, geometry,
# occupancy and launch code that decides how the kernel runs.
ROOFLINE_SOURCES = ("tma_kernels.cuh", "device_common.cuh", "params.h",
                    ("api.cu", "// ------------------------------------------------------------------ argument checks"))
NCU_TRAFFIC = {"sources_digest": "3a01f628d9696168", "variant": "sktma128x2w8", "N": 2048,
               "bytes_per_launch": 537185792 + 231728640}


# The other workloads of the path, each timed per shape and direction inside
# the same run (reported under "families"; not part of `value`):
# (name, op, dtype, M, row lengths, input distribution).
FAMILIES = (
    ("rms_1024x1024", "rms", "bf16", 1024, (1024,), "rms"),
    ("ln_16384", "ln", "bf16", 16384, (4096, 8192), "ln"),
    ("wide_rms_2048", "rms", "bf16", 2048, (16384, 32768, 65536, 131072), "rms"),
    ("wide_ln_2048", "ln", "bf16", 2048, (16384, 32768, 65536, 131072), "rms"),
) + tuple((f"llm_{op}_16384_{dt}", op, dt, 16384, (4096, 5120, 8192), "llm")
          for op in ("rms", "ln") for dt in ("bf16", "fp16", "fp32"))
# The general form (strided rows, a storage type per tensor, fused residual
# add), timed the same way: (name, op, x dtype, parameter dtype, y dtype, M, N,
# row stride, residual add).
EX_FAMILIES = (
    ("ex_rms_bf16_x_fp32_gamma", "rms", "bf16", "fp32", "bf16", 16384, 8192, 8192, False),
    ("ex_ln_bf16_x_fp32_gamma", "ln", "bf16", "fp32", "bf16", 16384, 8192, 8192, False),
    ("ex_rms_fp32_x_bf16_y", "rms", "fp32", "fp32", "bf16", 16384, 8192, 8192, False),
    ("ex_rms_bf16_strided", "rms", "bf16", "bf16", "bf16", 16384, 8192, 8448, False),
    ("ex_rms_bf16_residual", "rms", "bf16", "bf16", "bf16", 16384, 8192, 8192, True),
    ("ex_ln_bf16_residual", "ln", "bf16", "bf16", "bf16", 16384, 8192, 8192, True),
)
# Targets on the largest row length of each family (fraction of the measured
# copy peak): forward 0.85, backward 0.75.
TARGET = {"fwd": 0.85, "bwd": 0.75}
ESIZE = {"bf16": 2, "fp16": 2, "fp32": 4}
DTYPES_T = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def alg_bytes(op, direction, m, n, b):
    """Algorithmic bytes of one call: x, gamma, y, rstd (+ beta, mean) forward;
    dy, x, gamma, rstd, dx, dgamma (+ mean, dbeta) backward."""
    if direction == "fwd":
        return 2 * m * n * b + n * b + 4 * m if op == "rms" else 2 * m * n * b + 2 * n * b + 8 * m
    return 3 * m * n * b + n * b + 4 * m + 4 * n if op == "rms" else 3 * m * n * b + n * b + 8 * m + 8 * n


def fwd_bytes(m, n):
    return 2 * m * n * B + n * B + 4 * m


def bwd_bytes(m, n):
    return 3 * m * n * B + n * B + 4 * m + 4 * n


def kernel_digest(names=None, read=None) -> str:
    """Digest of the CUDA sources: all of them, or the listed entries (a file
    name, or (file name, marker) for the file's text before the marker)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rmsnorm_norm_fwd_gb300", "csrc")
    read = read or (lambda fn: open(os.path.join(csrc, fn), "rb").read())
    cut = {}
    for e in names or ():
        fn, mark = (e, None) if isinstance(e, str) else e
        cut[fn] = mark
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith((".cu", ".cuh", ".h", ".inc")) and (names is None or fn in cut):
            data = read(fn)
            if names is not None and cut[fn] is not None:
                data = data[:data.index(cut[fn].encode())]
            h.update(fn.encode() + data)
    return h.hexdigest()[:16]


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max_sum(vals_max, vals_sum, ws):
    """Max over ranks of vals_max, sum over ranks of vals_sum (gloo or nccl)."""
    if ws == 1:
        return vals_max, vals_sum
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    a = torch.tensor(vals_max, dtype=torch.float64, device=dev)
    b = torch.tensor(vals_sum, dtype=torch.float64, device=dev)
    dist.all_reduce(a, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return a.tolist(), b.tolist()


# ---------------------------------------------------------------------------- oracle on the host
def oracle_inputs(rows_per_n: int, seed: int = 20261202):
    """float64 host copies of `rows_per_n` rows of every N of the workload
    (drawn and promoted outside any timing)."""
    import numpy as np
    out = []
    for n in NS:
        inp = make_inputs(rows_per_n, n, dtype="bf16", dist="rms", op="rms", seed=seed)
        out.append((n, np.ascontiguousarray(inp.x.double().numpy()),
                    np.ascontiguousarray(inp.dy.double().numpy()),
                    np.ascontiguousarray(inp.gamma.double().numpy())))
    return out


def oracle_pass(data):
    """One timed pass of the fp64 oracle (as it stands) over `data`: forward
    plus backward (dx and dgamma) at every N.  Returns (bytes, seconds)."""
    import oracle
    tot_b, tot_t = 0, 0.0
    for n, x, dy, g in data:
        t0 = time.perf_counter()
        oracle.rmsnorm_fwd(x, g, EPS)
        oracle.rmsnorm_bwd(dy, x, g, EPS)
        tot_t += time.perf_counter() - t0
        tot_b += fwd_bytes(x.shape[0], n) + bwd_bytes(x.shape[0], n)
    return tot_b, tot_t


def cpu_baseline(target_s: float = 10.0):
    """The oracle on a bounded sample of the workload: `rows` rows at every N,
    timed repeatedly on all host threads (median pass; about target_s seconds
    of oracle time), and once on one thread for a per-core figure."""
    import oracle
    rows = 16384
    data = oracle_inputs(rows)
    th = oracle.threads()
    b, t = oracle_pass(data)
    reps = max(3, min(31, int(target_s / max(t, 1e-3))))
    ts = [t] + [oracle_pass(data)[1] for _ in range(reps - 1)]
    t_med = statistics.median(ts)
    one = oracle_inputs(1024)
    oracle.set_threads(1)
    try:
        b1, t1 = oracle_pass(one)
    finally:
        oracle.set_threads(th)
    return {"value": b / t_med / 1e9, "unit": "GB/s", "cores": th, "kind": "oracle",
            "sample": f"{rows} of {M} rows at each N of the sweep, fwd+bwd; median of {reps} passes "
                      f"({sum(ts):.1f} s of oracle time; bf16 inputs promoted to fp64 outside the timing)",
            "value_1_thread": b1 / t1 / 1e9,
            "sample_1_thread": f"1024 rows at each N, one pass on one thread ({t1:.1f} s)"}


def run_reference(args, ws, rank):
    """The oracle arm: the fp64 CPU oracle on the host cores, same workload,
    each step a bounded row sample of it."""
    if rank != 0:
        return
    import oracle
    rows = 4096
    data = oracle_inputs(rows)
    for _ in range(args.warmup):
        oracle_pass(data)
    tb, tt, th = 0, 0.0, oracle.threads()
    for _ in range(args.steps):
        b, t = oracle_pass(data)
        tb += b
        tt += t
    v = tb / tt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "N": list(NS), "sample_rows_per_N": rows},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": th, "kind": "oracle",
                             "sample": f"{rows} of {M} rows at each N per step, fwd+bwd"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- GPU arm
def run_ours(args, ws, rank, local):
    import rmsnorm_norm_fwd_gb300 as gb
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    # Inputs resident in HBM before timing.
    data = []
    for n in NS:
        inp = make_inputs(M, n, dtype="bf16", dist="rms", op="rms", seed=20261202 + rank)
        d = {"n": n, "x": inp.x.to(dev), "dy": inp.dy.to(dev), "gamma": inp.gamma.to(dev)}
        d["y"] = torch.empty_like(d["x"])
        d["dx"] = torch.empty_like(d["x"])
        d["rstd"] = torch.empty(M, device=dev, dtype=torch.float32)
        d["dgamma"] = torch.empty(n, device=dev, dtype=torch.float32)
        d["ws"] = torch.empty(gb.norm_bwd_workspace_size(False, M, n, torch.bfloat16), device=dev,
                              dtype=torch.uint8)
        d["host"] = inp
        data.append(d)
    scrub_w = torch.empty(L2_FLUSH_BYTES, device=dev, dtype=torch.uint8)
    scrub_r = torch.ones(L2_CLEAN_BYTES // 4, device=dev, dtype=torch.float32)

    def flush_l2():
        scrub_w.zero_()
        scrub_r.amax()

    def call_fwd(d):
        gb.rmsnorm_fwd(d["x"], d["gamma"], EPS, y=d["y"], rstd=d["rstd"])

    def call_bwd(d):
        gb.rmsnorm_bwd(d["dy"], d["x"], d["gamma"], d["rstd"], dx=d["dx"], dgamma=d["dgamma"],
                       workspace=d["ws"])

    def one_step(record):
        for d in data:
            flush_l2()
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            call_fwd(d)
            e1.record(stream)
            flush_l2()
            e1b = torch.cuda.Event(enable_timing=True)
            e1b.record(stream)
            call_bwd(d)
            e2.record(stream)
            if record is not None:
                record.append((d["n"], e0, e1, e1b, e2))

    for _ in range(max(3, args.warmup)):
        one_step(None)
    torch.cuda.synchronize()

    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    torch.cuda.synchronize()
    recs = []
    for _ in range(args.steps):
        one_step(recs)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None

    per = {}
    for n, e0, e1, e1b, e2 in recs:
        p = per.setdefault(n, {"fwd_ms": [], "bwd_ms": []})
        p["fwd_ms"].append(e0.elapsed_time(e1))
        p["bwd_ms"].append(e1b.elapsed_time(e2))
    t_local = sum(sum(p["fwd_ms"]) + sum(p["bwd_ms"]) for p in per.values())  # ms, all steps
    b_local = float(args.steps * sum(fwd_bytes(M, n) + bwd_bytes(M, n) for n in NS))
    (t_max,), (b_sum,) = reduce_max_sum([t_local], [b_local], ws)
    value = b_sum / (t_max * 1e-3) / 1e9

    # Dominant call: the largest share of the timed region.
    shares = []
    for n, p in per.items():
        for direction, key, nbytes in ((0, "fwd_ms", fwd_bytes(M, n)), (1, "bwd_ms", bwd_bytes(M, n))):
            shares.append((sum(p[key]), n, direction, nbytes, statistics.mean(p[key])))
    shares.sort(reverse=True)
    tot, n_dom, dir_dom, bytes_dom, avg_ms = shares[0]
    peak, peak_kind = peak_hbm()
    achieved = bytes_dom / (avg_ms * 1e-3) / 1e9
    vname = gb.variant_name(False, dir_dom, M, n_dom, torch.bfloat16)
    digest = kernel_digest()
    traffic = None
    if (NCU_TRAFFIC["sources_digest"] == kernel_digest(ROOFLINE_SOURCES) and NCU_TRAFFIC["N"] == n_dom
            and NCU_TRAFFIC["variant"] == vname):
        traffic = NCU_TRAFFIC["bytes_per_launch"]

    # End to end through the public API from pinned host memory, per step:
    # H2D of x, dy, gamma; forward; backward; D2H of y, rstd, dx, dgamma.
    # The host link is full duplex: shape i is computed on the launching
    # stream while shape i + 1 comes in on one copy stream and shape i - 1
    # goes out on another; events order every reuse of a buffer (a copy-in
    # waits for the previous step's computation on that shape, the
    # computation for the previous step's copy-out of its outputs).
    e2e = None
    if not args.no_e2e:
        hb = []
        for d in data:
            h = d["host"]
            hb.append({"x": h.x.pin_memory(), "dy": h.dy.pin_memory(), "gamma": h.gamma.pin_memory(),
                       "y": torch.empty_like(h.x).pin_memory(), "dx": torch.empty_like(h.x).pin_memory(),
                       "rstd": torch.empty(M, dtype=torch.float32).pin_memory(),
                       "dgamma": torch.empty(d["n"], dtype=torch.float32).pin_memory()})
        h2d = sum(h["x"].nbytes + h["dy"].nbytes + h["gamma"].nbytes for h in hb)
        d2h = sum(h["y"].nbytes + h["dx"].nbytes + h["rstd"].nbytes + h["dgamma"].nbytes for h in hb)

        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in data]
        ev_comp = [torch.cuda.Event() for _ in data]
        ev_out = [torch.cuda.Event() for _ in data]
        for i in range(len(data)):  # "previous step" events start completed
            ev_comp[i].record(stream)
            ev_out[i].record(stream)

        def e2e_step():
            start = torch.cuda.Event()
            start.record(stream)
            for i, (d, h) in enumerate(zip(data, hb)):
                s_in.wait_event(start)
                s_in.wait_event(ev_comp[i])  # the last step's kernels are done with x, dy, gamma
                with torch.cuda.stream(s_in):
                    d["x"].copy_(h["x"], non_blocking=True)
                    d["dy"].copy_(h["dy"], non_blocking=True)
                    d["gamma"].copy_(h["gamma"], non_blocking=True)
                ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                stream.wait_event(ev_out[i])  # the last step's outputs have left
                call_fwd(d)
                call_bwd(d)
                ev_comp[i].record(stream)
                s_out.wait_event(ev_comp[i])
                with torch.cuda.stream(s_out):
                    h["y"].copy_(d["y"], non_blocking=True)
                    h["dx"].copy_(d["dx"], non_blocking=True)
                    h["rstd"].copy_(d["rstd"], non_blocking=True)
                    h["dgamma"].copy_(d["dgamma"], non_blocking=True)
                ev_out[i].record(s_out)
            for e in ev_out:  # the step ends when its last output has arrived
                stream.wait_event(e)

        e2e_step()
        torch.cuda.synchronize()
        k2 = max(1, min(args.steps, 5))
        if dist:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(k2):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        (te,), (be,) = reduce_max_sum([a.elapsed_time(b)], [float(k2 * sum(
            fwd_bytes(M, n) + bwd_bytes(M, n) for n in NS))], ws)
        e2e = {"value": be / (te * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}

    families = None
    if rank == 0 and not args.no_families:
        fam_clock = ClockSampler(local)
        fam_clock.start()
        families = run_families(gb, dev, stream, flush_l2)
        families["rms_1024x1024"]["graph_100_calls"] = graph_per_call(gb, dev, stream, flush_l2)
        ex_fam = run_ex_families(gb, dev, stream, flush_l2)
        fam_clk = fam_clock.stop()
        # the sweep above, in the same form
        peak_, _ = peak_hbm()
        sweep = {}
        for n, p in sorted(per.items()):
            sweep[str(n)] = {d: {"gbs": round(nb / (statistics.median(p[k]) * 1e-3) / 1e9, 1),
                                 "frac": round(nb / (statistics.median(p[k]) * 1e-3) / 1e9 / peak_, 4),
                                 "ms": round(statistics.median(p[k]), 5),
                                 "variant": gb.variant_name(False, di, M, n, torch.bfloat16)}
                             for d, k, nb, di in (("fwd", "fwd_ms", fwd_bytes(M, n), 0),
                                                  ("bwd", "bwd_ms", bwd_bytes(M, n), 1))}
        big = sweep[str(NS[-1])]
        families = {"rms_sweep_65536": {"op": "rms", "dtype": "bf16", "M": M, "dist": "rms", "shapes": sweep,
                                        "largest": {"N": NS[-1], "fwd_frac": big["fwd"]["frac"],
                                                    "bwd_frac": big["bwd"]["frac"],
                                                    "meets_target": big["fwd"]["frac"] >= TARGET["fwd"]
                                                    and big["bwd"]["frac"] >= TARGET["bwd"]}},
                    **families, "general_form": ex_fam, "clocks": fam_clk,
                    "timing": "per shape and direction: median of 5 CUDA-event-timed calls after 3 "
                              "warm-up calls, L2 flushed before each; inputs drawn on the device; "
                              "rms_1024x1024 also as a CUDA graph of 100 calls on rotating buffers"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu = cpu_baseline(args.cpu_seconds)

    if rank == 0:
        breakdown = {str(n): {"fwd_gbs": round(fwd_bytes(M, n) / (statistics.median(p["fwd_ms"]) * 1e-3) / 1e9, 1),
                              "bwd_gbs": round(bwd_bytes(M, n) / (statistics.median(p["bwd_ms"]) * 1e-3) / 1e9, 1),
                              "fwd_variant": gb.variant_name(False, 0, M, n, torch.bfloat16),
                              "bwd_variant": gb.variant_name(False, 1, M, n, torch.bfloat16)}
                     for n, p in sorted(per.items())}
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "N": list(NS), "io_dtype": "bf16",
                       "l2": "flushed before every timed call: 1 GiB write then 512 MiB read, outside the events",
                       "timing": "CUDA events on the launching stream around each C-ABI call"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_kind": peak_kind,
                         "kernel": {"dir": "bwd" if dir_dom else "fwd", "N": n_dom, "variant": vname,
                                    "share_of_timed": tot / t_local,
                                    "note": ("backward time covers the row kernel and the column "
                                             "reduce of one call") if dir_dom else "one kernel"}},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * len(NS) * 3,
            "clocks": clocks,
            "breakdown": breakdown,
            "families": families,
            "kernel_digest": digest,
        }
        print(json.dumps(line), flush=True)


def run_families(gb, dev, stream, flush_l2, steps=5, warmup=3):
    """Every other workload of the path, per shape and direction: median
    CUDA-event time of `steps` calls (L2 flushed before each, outside the
    events), effective GB/s, fraction of the measured copy peak, and the
    variant that ran.  Inputs are drawn on the device with the same recipe."""
    peak, _ = peak_hbm()
    out = {}
    for name, op, dt, m, ns, dist in FAMILIES:
        ln, b = op == "ln", ESIZE[dt]
        shapes = {}
        for n in ns:
            inp = make_inputs(m, n, dtype=dt, dist=dist, op=op, device=str(dev))
            x, dy, g, be = inp.x, inp.dy, inp.gamma, inp.beta
            y, dx = torch.empty_like(x), torch.empty_like(x)
            mean, rstd = torch.empty(m, device=dev), torch.empty(m, device=dev)
            dg, db = torch.empty(n, device=dev), torch.empty(n, device=dev)
            wsb = torch.empty(gb.norm_bwd_workspace_size(ln, m, n, x.dtype), device=dev, dtype=torch.uint8)

            def fwd():
                if ln:
                    gb.layernorm_fwd(x, g, be, inp.eps, y=y, mean=mean, rstd=rstd)
                else:
                    gb.rmsnorm_fwd(x, g, inp.eps, y=y, rstd=rstd)

            def bwd():
                if ln:
                    gb.layernorm_bwd(dy, x, g, mean, rstd, dx=dx, dgamma=dg, dbeta=db, workspace=wsb)
                else:
                    gb.rmsnorm_bwd(dy, x, g, rstd, dx=dx, dgamma=dg, workspace=wsb)

            res = {}
            for d, call in (("fwd", fwd), ("bwd", bwd)):
                for _ in range(warmup):
                    flush_l2()
                    call()
                evs = []
                for _ in range(steps):
                    flush_l2()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    call()
                    e1.record(stream)
                    evs.append((e0, e1))
                torch.cuda.synchronize()
                ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
                gbs = alg_bytes(op, d, m, n, b) / (ms * 1e-3) / 1e9
                res[d] = {"gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "ms": round(ms, 5),
                          "variant": gb.variant_name(ln, 0 if d == "fwd" else 1, m, n, x.dtype)}
            shapes[str(n)] = res
            del inp, x, dy, g, be, y, dx, mean, rstd, dg, db, wsb
        big = shapes[str(ns[-1])]
        out[name] = {"op": op, "dtype": dt, "M": m, "dist": dist, "shapes": shapes,
                     "largest": {"N": ns[-1], "fwd_frac": big["fwd"]["frac"], "bwd_frac": big["bwd"]["frac"],
                                 "meets_target": big["fwd"]["frac"] >= TARGET["fwd"]
                                 and big["bwd"]["frac"] >= TARGET["bwd"]}}
    torch.cuda.empty_cache()
    return out


def ex_bytes(op, direction, m, n, bx, bp, by, residual):
    """Algorithmic bytes of one general-form call: forward x (+ residual in,
    h out), y, gamma (+ beta), rstd (+ mean); backward dy, x (h), dx
    (+ the residual gradient in), gamma, rstd (+ mean), dgamma (+ dbeta)."""
    ln = op == "ln"
    if direction == "fwd":
        return m * n * (bx + (2 * bx if residual else 0) + by) + n * bp * (2 if ln else 1) + 4 * m * (2 if ln else 1)
    return m * n * (by + bx + bx + (bx if residual else 0)) + n * bp + 4 * m * (2 if ln else 1) + \
        4 * n * (2 if ln else 1)


def run_ex_families(gb, dev, stream, flush_l2, steps=5, warmup=3):
    """The general form's workloads (EX_FAMILIES), per direction: median
    CUDA-event time, effective GB/s and fraction of the measured copy peak."""
    peak, _ = peak_hbm()
    out = {}
    for name, op, xd, pd, yd, m, n, ld, residual in EX_FAMILIES:
        ln = op == "ln"
        inp = make_inputs(m, n, dtype=xd, dist="llm", op=op, device=str(dev), param_dtype=pd, dy_dtype=yd)

        def rows(t):  # t inside a buffer of row stride ld
            buf = torch.empty(m, ld, device=dev, dtype=t.dtype)
            v = buf[:, :n]
            v.copy_(t)
            return v
        x, dy = rows(inp.x), rows(inp.dy)
        r = rows(make_inputs(m, n, dtype=xd, op=op, device=str(dev), seed=5).x) if residual else None
        dres = rows(make_inputs(m, n, dtype=xd, op=op, device=str(dev), seed=6).dy) if residual else None
        y, dx = rows(torch.empty(m, n, device=dev, dtype=DTYPES_T[yd])), rows(torch.empty_like(inp.x))
        h = rows(torch.empty_like(inp.x)) if residual else None
        g, be = inp.gamma, inp.beta if ln else None
        mean = torch.empty(m, device=dev) if ln else None
        rstd = torch.empty(m, device=dev)
        dg, db = torch.empty(n, device=dev), torch.empty(n, device=dev) if ln else None
        wsb = torch.empty(gb.norm_bwd_ex_workspace_size(ln, m, n), device=dev, dtype=torch.uint8)

        def fwd():
            gb.norm_fwd_ex(ln, x, g, be, inp.eps, residual=r, y=y, h=h, mean=mean, rstd=rstd)

        def bwd():
            gb.norm_bwd_ex(ln, dy, h if residual else x, g, mean, rstd, dres=dres, dx=dx, dgamma=dg, dbeta=db,
                           workspace=wsb)

        res = {"op": op, "x_dtype": xd, "param_dtype": pd, "y_dtype": yd, "M": m, "N": n, "row_stride": ld,
               "residual": residual}
        for d, call in (("fwd", fwd), ("bwd", bwd)):
            for _ in range(warmup):
                flush_l2()
                call()
            evs = []
            for _ in range(steps):
                flush_l2()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                evs.append((e0, e1))
            torch.cuda.synchronize()
            ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
            nb = ex_bytes(op, d, m, n, ESIZE[xd], ESIZE[pd], ESIZE[yd], residual)
            gbs = nb / (ms * 1e-3) / 1e9
            res[d] = {"gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "ms": round(ms, 5),
                      "variant": gb.ex_last_variant(0 if d == "fwd" else 1)}
        out[name] = res
        del inp, x, dy, r, dres, y, dx, h, wsb
    torch.cuda.empty_cache()
    return out


def graph_per_call(gb, dev, stream, flush_l2, m=1024, n=1024, calls=100):
    """RMSNorm bf16 [m, n], forward and backward, as the per-call time of a
    CUDA graph of `calls` back-to-back calls on rotating buffers (calls x the
    buffers of one call exceed L2, so every call reads its inputs from DRAM).
    A launch-bound shape's throughput when the launches are not in the way."""
    sets = []
    for i in range(calls):
        inp = make_inputs(m, n, dtype="bf16", op="rms", device=str(dev), seed=1000 + i)
        sets.append({"x": inp.x, "dy": inp.dy, "g": inp.gamma, "y": torch.empty_like(inp.x),
                     "dx": torch.empty_like(inp.x), "rstd": torch.empty(m, device=dev),
                     "dg": torch.empty(n, device=dev),
                     "ws": torch.empty(gb.norm_bwd_workspace_size(False, m, n, torch.bfloat16), device=dev,
                                       dtype=torch.uint8)})
    out = {}
    peak, _ = peak_hbm()
    for d in ("fwd", "bwd"):
        def body():
            for b in sets:
                if d == "fwd":
                    gb.rmsnorm_fwd(b["x"], b["g"], EPS, y=b["y"], rstd=b["rstd"])
                else:
                    gb.rmsnorm_bwd(b["dy"], b["x"], b["g"], b["rstd"], dx=b["dx"], dgamma=b["dg"],
                                   workspace=b["ws"])
        try:
            body()  # warm-up outside the capture (first-call set-up)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                body()
            ts = []
            for _ in range(5):
                flush_l2()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            us = statistics.median(ts) * 1e3 / calls
            nb = (fwd_bytes if d == "fwd" else bwd_bytes)(m, n)
            gbs = nb / (us * 1e-6) / 1e9
            out[d] = {"us_per_call": round(us, 3), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
        except Exception as e:  # a capture this torch build refuses: say so
            out[d] = {"error": f"{type(e).__name__}: {e}"[:200]}
    del sets
    torch.cuda.empty_cache()
    return out


def run_case(args):
    """One call shape of the workload, repeated: for profiling a single kernel
    (e.g. under ncu -k).  Prints one JSON line with the median CUDA-event time."""
    import rmsnorm_norm_fwd_gb300 as gb
    op, d, n = args.case.split(":")
    n, ln, bwd = int(n), op == "ln", d == "bwd"
    m = args.rows or M
    dt = args.dtype
    b = ESIZE[dt]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = make_inputs(m, n, dtype=dt, dist=args.dist or ("ln" if ln else "rms"), op=op, device="cuda")
    x, dy, g, be = inp.x, inp.dy, inp.gamma, inp.beta
    y, dx = torch.empty_like(x), torch.empty_like(x)
    mean, rstd = torch.empty(m, device=dev), torch.empty(m, device=dev)
    dg, db = torch.empty(n, device=dev), torch.empty(n, device=dev)
    ws = torch.empty(gb.norm_bwd_workspace_size(ln, m, n, x.dtype), device=dev, dtype=torch.uint8)

    def fwd():
        if ln:
            gb.layernorm_fwd(x, g, be, inp.eps, y=y, mean=mean, rstd=rstd)
        else:
            gb.rmsnorm_fwd(x, g, inp.eps, y=y, rstd=rstd)

    def bwd_():
        if ln:
            gb.layernorm_bwd(dy, x, g, mean, rstd, dx=dx, dgamma=dg, dbeta=db, workspace=ws)
        else:
            gb.rmsnorm_bwd(dy, x, g, rstd, dx=dx, dgamma=dg, workspace=ws)

    if args.variant:
        gb.force_variant(ln, int(bwd), x.dtype, args.variant)
    fwd()
    call = bwd_ if bwd else fwd
    for _ in range(args.warmup):
        call()
    stream = torch.cuda.current_stream(dev)
    ts = []
    for _ in range(args.steps):
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        e.record(stream)
        e.synchronize()
        ts.append(a.elapsed_time(e))
    ms = statistics.median(ts)
    nbytes = alg_bytes(op, d, m, n, b)
    print(json.dumps({"case": args.case, "dtype": dt, "M": m, "N": n,
                      "variant": gb.variant_name(ln, int(bwd), m, n, x.dtype),
                      "ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9, "l2": "not flushed"}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline leg")
    ap.add_argument("--no-families", action="store_true",
                    help="skip the per-shape timing of the other workloads")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--case", help="op:dir:N (e.g. rms:bwd:2048): time one call shape of bf16 rows "
                                   "only, for profiling one kernel")
    ap.add_argument("--rows", type=int, default=0, help="rows for --case (default 65536)")
    ap.add_argument("--variant", help="with --case: force this kernel variant (profiling)")
    ap.add_argument("--dtype", default="bf16", choices=("bf16", "fp16", "fp32"), help="with --case")
    ap.add_argument("--dist", default=None, choices=("rms", "ln", "llm"), help="with --case")
    args = ap.parse_args(argv)
    if args.case:
        run_case(args)
        return
    args.warmup = max(3, args.warmup)

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank)
        else:
            if not torch.cuda.is_available():
                raise SystemExit("bench.py: no CUDA device; the GPU arm needs one")
            run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

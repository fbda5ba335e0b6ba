"""Seeded synthetic inputs shared by the CUDA path and the fp64 oracle.

This module holds no normalisation arithmetic: it only draws random tensors.
Both sides of every parity check read the same host tensors, so the oracle
sees exactly the dtype-rounded values the kernels see.

Recipe (one ``torch.Generator`` per tensor, seeded from ``seed`` and the
tensor's slot, so adding a tensor never shifts another's draws; on the CPU for
every parity check, optionally on the GPU for timing runs, where the same
recipe gives other draws of the same distributions):
  * draw in float32, apply the distribution, then round once to the dtype;
  * ``dist="rms"``:  x ~ N(0, 1)
  * ``dist="ln"``:   x ~ N(0.5, 2^2)
  * ``dist="llm"``:  x ~ N(0, 1), then 1% of rows (seeded choice) scaled by
    100, then 0.1% of all elements (seeded choice, anywhere) set to +-60 with
    a random sign -- an accumulation stress for fp16/bf16 rows;
  * gamma = 1 + 0.1 * N(0, 1), beta = 0.1 * N(0, 1), dy ~ N(0, 1) for all.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

DEFAULT_SEED = 20261202

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}

# Tensor slots: each tensor draws from its own generator.
_SLOT = {"x": 0, "gamma": 1, "beta": 2, "dy": 3, "rows": 4, "elems": 5, "signs": 6}


def _gen(seed: int, slot: str, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + _SLOT[slot])
    return g


@dataclass
class NormInputs:
    x: torch.Tensor        # [M, N] in dtype, CPU
    gamma: torch.Tensor    # [N] in dtype, CPU
    beta: torch.Tensor     # [N] in dtype, CPU
    dy: torch.Tensor       # [M, N] in dtype, CPU
    eps: float
    dtype: str
    dist: str


def default_eps(op: str) -> float:
    """1e-6 for RMSNorm and 1e-5 for LayerNorm, the values of the workloads."""
    return 1e-6 if op == "rms" else 1e-5


def make_inputs(M: int, N: int, dtype: str = "bf16", dist: str = "rms", op: str = "rms",
                seed: int = DEFAULT_SEED, eps: float | None = None,
                with_dy: bool = True, device: str = "cpu", param_dtype: str | None = None,
                dy_dtype: str | None = None) -> NormInputs:
    """Draw one seeded problem of shape [M, N] (see the module docstring).
    device: where the draws happen and the tensors live ("cpu" for anything the
    oracle reads).  gamma / beta are rounded to param_dtype and dy to dy_dtype
    (default: dtype, the type of x)."""
    t = DTYPES[dtype]
    tp = DTYPES[param_dtype or dtype]
    td = DTYPES[dy_dtype or dtype]
    dev = torch.device(device)
    gen = (lambda slot: _gen(seed, slot, dev.type if dev.type == "cpu" else str(dev)))
    x = torch.randn(M, N, generator=gen("x"), dtype=torch.float32, device=dev)
    if dist == "ln":
        x = x * 2.0 + 0.5
    elif dist == "llm":
        n_rows = max(1, (M + 99) // 100) if M > 0 else 0
        if n_rows:
            rows = torch.randperm(M, generator=gen("rows"), device=dev)[:n_rows]
            x[rows] *= 100.0
        n_el = (M * N) // 1000
        if n_el:
            flat = x.view(-1)
            idx = torch.randint(0, M * N, (n_el,), generator=gen("elems"), device=dev)
            sgn = torch.randint(0, 2, (n_el,), generator=gen("signs"), device=dev).float() * 2.0 - 1.0
            flat[idx] = 60.0 * sgn
    elif dist != "rms":
        raise ValueError(f"unknown dist {dist!r}")
    gamma = 1.0 + 0.1 * torch.randn(N, generator=gen("gamma"), dtype=torch.float32, device=dev)
    beta = 0.1 * torch.randn(N, generator=gen("beta"), dtype=torch.float32, device=dev)
    if with_dy:
        dy = torch.randn(M, N, generator=gen("dy"), dtype=torch.float32, device=dev).to(td)
    else:
        dy = torch.empty(0, dtype=td, device=dev)
    return NormInputs(x=x.to(t), gamma=gamma.to(tp), beta=beta.to(tp), dy=dy,
                      eps=default_eps(op) if eps is None else float(eps), dtype=dtype, dist=dist)

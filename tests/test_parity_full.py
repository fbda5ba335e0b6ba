"""CUDA path vs the fp64 oracle at the full workload sizes, in the launch
configuration the benchmark times (default dispatch).  y, rstd, mean and dx
are checked on sampled rows (first, last, 62 seeded ones and, for the
accumulation-stress inputs, every row scaled by 100); dgamma and dbeta against
the oracle's full column sums over all rows (GPU)."""
import pytest

from parity_util import run_case

pytestmark = pytest.mark.gpu

WORKLOADS = (
    # RMSNorm, 1024 x 1024 bf16: the small single-shape case (every row checked)
    [("rms", "bf16", 1024, 1024, "rms", False)]
    # RMSNorm big-M small-N sweep, bf16
    + [("rms", "bf16", 65536, n, "rms", True) for n in (256, 384, 512, 768, 1024, 2048)]
    # LayerNorm with gamma and beta, x ~ N(0.5, 2^2), bf16
    + [("ln", "bf16", 16384, n, "ln", True) for n in (4096, 8192)]
    # wide rows, RMSNorm and LayerNorm, bf16
    + [(op, "bf16", 2048, n, "rms", True) for op in ("rms", "ln") for n in (16384, 32768, 65536, 131072)]
    # LLM-shaped rows with outliers, three dtypes
    + [(op, dt, 16384, n, "llm", True) for op in ("rms", "ln") for dt in ("bf16", "fp16", "fp32")
       for n in (4096, 5120, 8192)]
)


@pytest.mark.parametrize("op,dtype,M,N,dist,sampled", WORKLOADS,
                         ids=[f"{o}-{d}-{m}x{n}-{s}" for o, d, m, n, s, _ in WORKLOADS])
def test_workload(op, dtype, M, N, dist, sampled):
    rep, _, _ = run_case(op, dtype, M, N, dist=dist, rows="sample" if sampled else None)
    rep.assert_ok()

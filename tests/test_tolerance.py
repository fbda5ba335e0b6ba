"""The parity machinery itself, on the CPU: the bounds come from the oracle and
fp32 arithmetic only, accept the oracle's own values rounded to the output
dtype, reject a planted error just above the stated figure, and the sampled
rows of a full-size check include every row of the accumulation-stress recipe
scaled by 100."""
import numpy as np
import pytest
import re

import torch

import oracle
from parity_util import compare, row_threads, sample_rows, sum_depth, ulp
from rmsnorm_norm_fwd_gb300.inputs import DTYPES, make_inputs


def _as_gpu_out(op, inp):
    """The oracle's results rounded to what the kernels store: y, dx in the
    dtype, statistics and parameter sums in fp32."""
    t = DTYPES[inp.dtype]
    if op == "rms":
        y, r = oracle.rmsnorm_fwd(inp.x, inp.gamma, inp.eps)
        dx, dg = oracle.rmsnorm_bwd(inp.dy, inp.x, inp.gamma, inp.eps)
        return {"y": torch.from_numpy(y).to(t), "rstd": torch.from_numpy(r).float(),
                "dx": torch.from_numpy(dx).to(t), "dgamma": torch.from_numpy(dg).float()}
    y, m, r = oracle.layernorm_fwd(inp.x, inp.gamma, inp.beta, inp.eps)
    dx, dg, db = oracle.layernorm_bwd(inp.dy, inp.x, inp.gamma, inp.eps)
    return {"y": torch.from_numpy(y).to(t), "mean": torch.from_numpy(m).float(),
            "rstd": torch.from_numpy(r).float(), "dx": torch.from_numpy(dx).to(t),
            "dgamma": torch.from_numpy(dg).float(), "dbeta": torch.from_numpy(db).float()}


VARIANTS = {"rms": ("s256x4b256m4", "tmp256x4b512"), "ln": ("tmp256x4b512", "bwide512u4c2p1f0m1")}


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_rounded_oracle_passes(op, dtype):
    inp = make_inputs(40, 512, dtype=dtype, dist="llm", op=op)
    rep = compare(op, inp, _as_gpu_out(op, inp), variants=VARIANTS[op])
    rep.assert_ok()
    # a correctly rounded result needs no floor anywhere (torch may round
    # fp64 -> fp16 through fp32: a hair above half an ulp)
    assert rep.stats["dx"]["max_ulps"] <= 0.501
    assert rep.stats["y"]["n_floor_only"] == 0 and rep.stats["dx"]["n_floor_only"] == 0


@pytest.mark.parametrize("op", ["rms", "ln"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_planted_dx_error_fails(op, dtype):
    """Three output ulps on one large dx element exceed the stated 2 ulps plus
    every fp32 floor term (tiny next to a bf16/fp16 ulp)."""
    inp = make_inputs(40, 512, dtype=dtype, op=op)
    out = _as_gpu_out(op, inp)
    dx = out["dx"].double()
    i = int(torch.argmax(dx.abs().flatten()))
    v = dx.flatten()[i].item()
    out["dx"].view(-1)[i] = torch.tensor(v + 3 * float(ulp(np.array([v]), dtype)[0])).to(DTYPES[dtype])
    rep = compare(op, inp, out, variants=VARIANTS[op])
    assert not rep.ok and rep.stats["dx"]["n_bad"] == 1


@pytest.mark.parametrize("op", ["rms", "ln"])
def test_planted_rstd_error_fails(op):
    """rstd off by 1e-5 relative breaks both the stated figure and the a-priori
    bound the y and dx checks rely on."""
    inp = make_inputs(40, 512, dtype="fp32", op=op)
    out = _as_gpu_out(op, inp)
    out["rstd"][3] *= 1 + 2e-5
    rep = compare(op, inp, out, variants=VARIANTS[op])
    assert not rep.ok and rep.stats["rstd"]["n_bad"] == 1 and rep.stats["rstd_apriori"]["n_bad"] == 1


def test_sum_depth_from_geometry():
    # 512 threads share a row of 8192 bf16 elements: 16 serial, 5 shuffle
    # levels, 16 warps, + 4
    assert sum_depth(8192, "tmp512x4b512", "bf16") == 16 + 5 + 16 + 4
    # a cluster of 8 CTAs of 256 threads, 131072 bf16: 64 serial, 5, 8, 8, + 4
    assert sum_depth(131072, "bwide256u4c8p1f0m2", "bf16") == 64 + 5 + 8 + 8 + 4
    # element-wise: 256 threads, one element each per 256
    assert sum_depth(1000, "elem", "fp32") == 4 + 5 + 8 + 4
    # a row shorter than the row group: still whole vectors per thread
    assert sum_depth(264, "32x4r1c1b256", "bf16") == 16 + 5 + 4
    with pytest.raises(ValueError):
        row_threads("nonsense")


def test_every_dispatched_variant_has_a_depth():
    import os
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(__file__)), "rmsnorm_norm_fwd_gb300", "csrc",
                        "dispatch_table.inc")
    names = re.findall(r'"([^"]+)"\}', open(path).read())
    assert names
    for n in names:
        row_threads(n)


def test_sample_includes_scaled_rows():
    inp = make_inputs(3000, 64, dtype="bf16", dist="llm")
    rows = sample_rows(3000, x=inp.x)
    ms = (inp.x.float() ** 2).mean(dim=1)
    scaled = set(torch.nonzero(ms > 400.0).flatten().tolist())
    assert len(scaled) == 30 and scaled <= set(rows.tolist())


def test_general_form_names_parse():
    """Every general-form kernel the library holds has a name row_threads reads
    (the tests derive each call's tolerance from the name of the kernel that
    ran, as gbnorm_ex_last_variant reports it)."""
    import rmsnorm_norm_fwd_gb300 as g
    from parity_util import row_threads
    for ln in (False, True):
        for d in (0, 1):
            names = g.ex_variants(ln, d)
            assert names[-1] == "exe" and len(names) == len(set(names)) > 1
            for name in names:
                tpr, cl, elem = row_threads(name)
                assert cl == 1 and elem == (name == "exe")
                m = re.fullmatch(r"exr?[fb](\d+)x(\d+)b(\d+)(?:_(?:bf16|fp16|fp32))?", name)
                assert elem or (m and int(m.group(1)) == tpr and int(m.group(3)) % tpr == 0)

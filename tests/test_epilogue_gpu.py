"""GPU parity of the output epilogue (RMSNorm, gain, SiLU output gate) through
the C ABI against the float64 oracle.

Bar, element by element on the same seeded inputs: max|d| / max|ref| <= 2e-2
for bf16 rows and <= 1e-4 for fp32 rows (the forward's bar), and every element
within a rounding-sized band of its own reference: 1e-2 |ref| for bf16 (one
bf16 rounding of y is at most 2^-9 |y|) and 1e-5 |ref| for fp32.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_10_gb300 as gdr
from gated_delta_rule_10_gb300 import workloads as wl
from oracle import epilogue as oep
from tests.gdr_testutil import TOL, f64, gpu_forward, rel_err

pytestmark = pytest.mark.gpu

ELEM_RTOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}
EPS = 1e-6


def run(x, eps=EPS, out=None):
    d = {k: v.cuda() for k, v in x.items()}
    if out == "o":
        y = gdr.rmsnorm_gate(d["o"], d["z"], d["weight"], eps, out=d["o"])
    elif out == "z":
        y = gdr.rmsnorm_gate(d["o"], d["z"], d["weight"], eps, out=d["z"])
    else:
        y = gdr.rmsnorm_gate(d["o"], d["z"], d["weight"], eps)
    torch.cuda.synchronize()
    return y.cpu()


def compare(y, x, eps=EPS, rows=None):
    o, z = x["o"], x["z"]
    if rows is not None:
        y, o, z = y[rows], o[rows], z[rows]
    ref = oep.rmsnorm_gate(f64(o), f64(z), f64(x["weight"]), eps)
    got = f64(y)
    assert rel_err(got, ref) <= TOL[x["o"].dtype]
    band = ELEM_RTOL[x["o"].dtype] * np.abs(ref) + 1e-7 * np.max(np.abs(ref))
    bad = np.abs(got - ref) > band
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("dv", [64, 128, 256])
@pytest.mark.parametrize("rows", [1, 3, 37, 4099])
def test_epilogue_matches_oracle(dtype, dv, rows):
    x = wl.epilogue_inputs(rows, dv, dtype, seed=rows + dv)
    compare(run(x), x)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("where", ["o", "z"])
def test_epilogue_in_place(dtype, where):
    x = wl.epilogue_inputs(517, 128, dtype, seed=3)
    y = run(x, out=where)
    compare(y, x)
    assert torch.equal(y, run(x))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_epilogue_degenerate_rows(dtype):
    # a zero row (eps keeps it finite: y = 0), a constant row, a row scaled by
    # 1e3, large-magnitude gates on both sides (silu -> z and -> 0)
    x = wl.epilogue_inputs(8, 128, dtype, seed=5)
    o, z = x["o"].clone(), x["z"].clone()
    o[0] = 0
    o[1] = 0.25
    o[2] = o[3] * 1000
    z[4] = 40.0
    z[5] = -40.0
    x = {"o": o, "z": z, "weight": x["weight"]}
    y = run(x, eps=1e-5)
    compare(y, x, eps=1e-5)
    assert torch.all(y[0] == 0)
    assert torch.all(y[5].abs() < 1e-12)


def test_epilogue_empty_input_is_a_no_op():
    o = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, device="cuda")
    assert gdr.rmsnorm_gate(o, o.clone(), w).numel() == 0


def test_epilogue_on_the_forward_output_full_size():
    # the 4 x 4096 x 16 x 128 bf16 read-out of the Gated DeltaNet workload as
    # the benchmark runs it; sampled rows against the oracle
    c = wl.CONFIGS[2]
    o, _ = gpu_forward(wl.config_inputs(2))
    rows = c["B"] * c["T"] * c["H"]
    e = wl.epilogue_inputs(rows, c["dv"], torch.bfloat16, seed=11)
    xe = {"o": o.reshape(rows, c["dv"]).cpu(), "z": e["z"], "weight": e["weight"]}
    y = run(xe)
    gen = np.random.default_rng(0)
    sample = np.concatenate([gen.choice(rows, 4096, replace=False), [0, rows - 1]])
    compare(y, xe, rows=torch.from_numpy(sample))

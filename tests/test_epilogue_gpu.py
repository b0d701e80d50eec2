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


# ------------------------------------------------ fused into the chunked forward
def _gate_inputs(x, seed):
    B, T, H = x["q"].shape[:3]
    dv = x["v"].shape[-1]
    e = wl.epilogue_inputs(B * T * H, dv, x["q"].dtype, seed=seed)
    return e["z"].reshape(B, T, H, dv), e["weight"]


def _fused_oracle(x, z, weight, eps=EPS, heads_per_group=8):
    """Oracle forward (float64 token recurrence) followed by the oracle epilogue,
    over groups of heads; returns (y, hT) as float64 arrays."""
    from tests.gdr_testutil import oracle_forward, select
    B, T, H = x["q"].shape[:3]
    ys, hs = [], []
    for h0 in range(0, H, heads_per_group):
        idx = list(range(h0, min(H, h0 + heads_per_group)))
        ro, rh = oracle_forward(select(x, heads=idx))
        ys.append(oep.rmsnorm_gate(ro, f64(z[:, :, idx]), f64(weight), eps))
        hs.append(rh)
    return np.concatenate(ys, axis=2), np.concatenate(hs, axis=1)


@pytest.mark.parametrize("variant", ["gdn", "qdelta", "kda", "gdn2"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 65, 200])
def test_fused_epilogue_matches_forward_then_epilogue_oracle(variant, dk, dv, T):
    """gdr_chunk_fwd_gated (fused in the state pass at d_k = d_v = 128, the forward
    then the epilogue kernel otherwise) against the oracle forward followed by
    the oracle epilogue, every element."""
    x = wl.make_inputs(variant, 2, T, 3, dk, dv, torch.bfloat16, seed=T + dk + dv, h0_std=0.02)
    z, weight = _gate_inputs(x, seed=T + 1)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    y, hT = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"], d["b"], d["w"],
                          d["h0"], scale=x["scale"], flags=x["flags"],
                          out_gate=(z.cuda(), weight.cuda(), EPS))
    torch.cuda.synchronize()
    ry, rh = _fused_oracle(x, z, weight)
    assert rel_err(y.float().cpu(), ry) <= TOL[torch.bfloat16]
    assert rel_err(hT.cpu(), rh) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("pipeline", [1, 4])
def test_fused_epilogue_pipelined_and_plain_agree(pipeline):
    """The fused epilogue through the plain and the pipelined call, against the
    oracle (a long sequence so that the pipelined call has several segments)."""
    x = wl.make_inputs("gdn2", 1, 64 * 40 + 17, 4, 128, 128, torch.bfloat16, seed=8,
                       h0_std=0.02)
    z, weight = _gate_inputs(x, seed=12)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    y, hT = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"], d["b"], d["w"],
                          d["h0"], scale=x["scale"], flags=x["flags"], pipeline=pipeline,
                          out_gate=(z.cuda(), weight.cuda(), EPS))
    torch.cuda.synchronize()
    ry, rh = _fused_oracle(x, z, weight)
    assert rel_err(y.float().cpu(), ry) <= TOL[torch.bfloat16]
    assert rel_err(hT.cpu(), rh) <= TOL[torch.bfloat16]


def test_fused_epilogue_gated_deltanet2_workload_every_sequence():
    """The Gated DeltaNet-2 prefill (1 x 65536 x 32 x 128 bf16) through the
    pipelined call the benchmark times, epilogue fused; every element of y of
    every (batch, head) against the oracle forward and epilogue."""
    c = wl.CONFIGS[5]
    x = wl.config_inputs(5, gen_device="cuda")
    B, T, H, dv = c["B"], c["T"], c["H"], c["dv"]
    e = wl.epilogue_inputs(B * T * H, dv, c["dtype"], seed=11, device="cuda")
    z, weight = e["z"].reshape(B, T, H, dv), e["weight"]
    shape = gdr.make_shape(B, T, H, c["dk"], dv, c["dtype"], x["flags"], x["scale"])
    y, hT = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["b"], x["w"],
                          x["h0"], scale=x["scale"], flags=x["flags"],
                          pipeline=gdr.pipeline_segments(shape), out_gate=(z, weight, EPS))
    torch.cuda.synchronize()
    from tests.gdr_testutil import ErrAcc, oracle_forward, select
    ey, eh = ErrAcc(), ErrAcc()
    for h0 in range(0, H, 8):
        idx = list(range(h0, h0 + 8))
        ro, rh = oracle_forward(select(x, heads=idx))
        ey.add(y[:, :, h0:h0 + 8].float().cpu(),
               oep.rmsnorm_gate(ro, f64(z[:, :, h0:h0 + 8]), f64(weight), EPS))
        eh.add(hT[:, h0:h0 + 8].cpu(), rh)
    assert ey.value() <= TOL[torch.bfloat16] and eh.value() <= TOL[torch.bfloat16], (
        ey.value(), eh.value())

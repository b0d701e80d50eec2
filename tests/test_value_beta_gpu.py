"""GPU parity of the write strength per value channel (GDR_BETA_CHANNEL, the
README variant of the LLMs-from-scratch Gated DeltaNet chapter, section 11.3)
through the C ABI against the float64 oracle.

Two paths: bf16 inputs with the full workspace take the two-kernel chunked
path (per-column substitution); fp32 inputs, the minimum workspace and the
decode step take the token-order scan.

Bar, element by element on the same seeded inputs: max|d| / max|ref| <= 2e-2
for bf16 inputs and 1e-4 for fp32 inputs, for o and the final state. The
token-order scan keeps the state in fp32 and rounds only o, so there the final
state is also held to 1e-4 with bf16 inputs, and fp32 o to 1e-5.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_10_gb300 as gdr
from gated_delta_rule_10_gb300 import workloads as wl
from tests.gdr_testutil import (TOL, f64, full_parity, gpu_forward, oracle_forward, rel_err,
                                select, to_dev)

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.bfloat16]


def check(x, token):
    """token: the token-order scan (minimum workspace), else the default path."""
    o, hT = gpu_forward(x, single_kernel=token)
    torch.cuda.synchronize()
    ro, rh = oracle_forward(x)
    eo, eh = rel_err(o.float().cpu(), ro), rel_err(hT.cpu(), rh)
    f32 = x["q"].dtype == torch.float32
    if token or f32:
        assert eo <= (1e-5 if f32 else TOL[torch.bfloat16]), eo
        assert eh <= 1e-4, eh
    else:
        assert eo <= TOL[torch.bfloat16] and eh <= TOL[torch.bfloat16], (eo, eh)
    return eo, eh


@pytest.mark.parametrize("dtype", DTYPES, ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 31, 32, 33, 100])
def test_value_beta_small_shapes_token_scan(T, dk, dv, dtype):
    x = wl.make_inputs("vbeta", 2, T, 3, dk, dv, dtype, seed=T + dk + 3 * dv, h0_std=0.05)
    check(x, token=True)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 64 * 9 + 7])
def test_value_beta_small_shapes_chunked(T, dk, dv):
    x = wl.make_inputs("vbeta", 2, T, 3, dk, dv, torch.bfloat16, seed=T + dk + 5 * dv,
                       h0_std=0.05)
    check(x, token=False)


def test_value_beta_paths_agree():
    x = wl.make_inputs("vbeta", 2, 333, 4, 128, 128, torch.bfloat16, seed=71, h0_std=0.02)
    o1, h1 = gpu_forward(x)
    o2, h2 = gpu_forward(x, single_kernel=True)
    torch.cuda.synchronize()
    assert rel_err(o1.float().cpu(), o2.float().cpu().double().numpy()) <= TOL[torch.bfloat16]
    assert rel_err(h1.cpu(), h2.cpu().double().numpy()) <= TOL[torch.bfloat16]


def test_value_beta_zero_state_no_final_state():
    x = wl.make_inputs("vbeta", 1, 77, 2, 128, 128, torch.bfloat16, seed=9)
    o, hT = gpu_forward(x, output_final_state=False)
    assert hT is None
    ro, _ = oracle_forward(x)
    assert rel_err(o.float().cpu(), ro) <= TOL[torch.bfloat16]


def test_value_beta_streaming_split_in_place():
    """Two calls with h0 and hT the same buffer equal one call over both halves."""
    x = wl.make_inputs("vbeta", 2, 150, 2, 128, 128, torch.float32, seed=12, h0_std=0.05)
    d = to_dev(x)
    state = d["h0"].clone()
    outs = []
    for sl in (slice(0, 61), slice(61, 150)):
        part = {n: (d[n][:, sl].contiguous() if n in ("q", "k", "v", "g", "beta") else None)
                for n in ("q", "k", "v", "g", "beta")}
        o, _ = gdr.chunk_fwd(part["q"], part["k"], part["v"], part["g"], part["beta"], h0=state,
                             hT=state, scale=x["scale"], flags=x["flags"])
        outs.append(o)
    torch.cuda.synchronize()
    ro, rh = oracle_forward(x)
    assert rel_err(torch.cat(outs, 1).cpu(), ro) <= 1e-5
    assert rel_err(state.cpu(), rh) <= 1e-5


@pytest.mark.parametrize("dtype", DTYPES, ids=["f32", "bf16"])
def test_value_beta_decode_step(dtype):
    """gdr_recurrent_step under the flag: one token, the state updated in place."""
    N, H, dk, dv = 5, 3, 128, 64
    y = wl.make_inputs("vbeta", N, 1, H, dk, dv, dtype, seed=21, h0_std=0.05)
    d = to_dev(y)
    state = d["h0"].clone()
    o = gdr.recurrent_step(d["q"][:, 0], d["k"][:, 0], d["v"][:, 0], d["g"][:, 0], state,
                           d["beta"][:, 0], scale=y["scale"], flags=y["flags"])
    torch.cuda.synchronize()
    ro, rh = oracle_forward(y)
    assert rel_err(o.float().cpu().unsqueeze(1), ro) <= (1e-5 if dtype == torch.float32
                                                         else TOL[torch.bfloat16])
    assert rel_err(state.cpu(), rh) <= 1e-4


def test_value_beta_equal_gate_matches_gated_deltanet_path():
    """With beta equal across value channels the flag reproduces plain Gated
    DeltaNet, here against the chunked bf16 path (each within the bar)."""
    x = wl.make_inputs("gdn", 2, 200, 2, 128, 128, torch.bfloat16, seed=31, h0_std=0.02)
    xv = dict(x)
    xv["beta"] = x["beta"][..., None].expand(*x["beta"].shape, 128).contiguous()
    xv["flags"] = wl.BETA_CHANNEL
    o1, h1 = gpu_forward(x)
    o2, h2 = gpu_forward(xv)
    torch.cuda.synchronize()
    assert rel_err(o2.float().cpu(), o1.float().cpu().double().numpy()) <= TOL[torch.bfloat16]
    assert rel_err(h2.cpu(), h1.cpu().double().numpy()) <= TOL[torch.bfloat16]


def test_value_beta_workload_full_size_every_sequence():
    """4 x 4096 x 16 x 128 bf16 as the benchmark runs it; every (batch, head)."""
    x = wl.config_inputs("vbeta", gen_device="cuda")
    o, hT = gpu_forward(x)
    torch.cuda.synchronize()
    eo, eh = full_parity(x, o, hT)
    assert eo <= TOL[torch.bfloat16] and eh <= TOL[torch.bfloat16], (eo, eh)

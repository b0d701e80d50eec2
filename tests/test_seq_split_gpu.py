"""GPU parity of the sequence split (gdr_chunk_fwd_split, and gdr_chunk_fwd's
default policy when B * H is small) against the float64 oracle.

Same bar as the unsplit path: max|d| / max|ref| <= 2e-2 (bf16) for o and the
final state, element by element on the same seeded inputs.
"""
import pytest
import torch

import gated_delta_rule_10_gb300 as gdr
from gated_delta_rule_10_gb300 import workloads as wl
from tests.gdr_testutil import TOL, oracle_forward, rel_err, select, to_dev

pytestmark = pytest.mark.gpu

VARIANTS = ["gdn", "qdelta", "kda", "gdn2"]
BAR = TOL[torch.bfloat16]


def split_forward(x, segments=None, output_final_state=True):
    d = to_dev(x)
    shape = gdr.make_shape(*d["q"].shape, d["v"].shape[-1], d["q"].dtype, x["flags"], x["scale"])
    n = gdr.chunk_fwd_workspace_bytes(shape, segments=segments)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    o, hT = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"], d["b"], d["w"],
                          d["h0"], scale=x["scale"], flags=x["flags"], workspace=ws,
                          segments=segments, output_final_state=output_final_state)
    gdr.chunk_fwd_check(ws)
    return o, hT


def check(x, **kw):
    o, hT = split_forward(x, **kw)
    torch.cuda.synchronize()
    ro, rh = oracle_forward(x)
    eo = rel_err(o.float().cpu(), ro)
    assert eo <= BAR, eo
    if hT is not None:
        eh = rel_err(hT.cpu(), rh)
        assert eh <= BAR, eh


@pytest.mark.parametrize("segments", [2, 3, 5])
@pytest.mark.parametrize("variant", VARIANTS)
def test_split_every_variant(variant, segments):
    x = wl.make_inputs(variant, 2, 64 * 9 + 17, 3, 128, 128, torch.bfloat16, seed=40 + segments,
                       h0_std=0.05)
    check(x, segments=segments)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128)])
def test_split_widths(dk, dv):
    x = wl.make_inputs("gdn2", 2, 64 * 7 + 5, 2, dk, dv, torch.bfloat16, seed=dk + dv, h0_std=0.05)
    check(x, segments=3)


def test_split_more_runs_than_chunks_and_no_states():
    x = wl.make_inputs("kda", 1, 100, 2, 128, 128, torch.bfloat16, seed=3)   # 2 chunks
    check(x, segments=4)
    check(x, segments=4, output_final_state=False)


def test_split_and_unsplit_agree():
    x = wl.make_inputs("gdn", 2, 64 * 12, 2, 128, 128, torch.bfloat16, seed=8, h0_std=0.02)
    o1, h1 = split_forward(x, segments=1)
    o4, h4 = split_forward(x, segments=4)
    torch.cuda.synchronize()
    assert rel_err(o4.float().cpu(), o1.float().cpu().double().numpy()) <= BAR
    assert rel_err(h4.cpu(), h1.cpu().double().numpy()) <= BAR


def test_default_policy_splits_few_long_sequences():
    x = wl.make_inputs("gdn2", 1, 64 * 160 + 23, 2, 128, 128, torch.bfloat16, seed=17,
                       h0_std=0.02)
    d = to_dev(x)
    shape = gdr.make_shape(*d["q"].shape, 128, torch.bfloat16, x["flags"], x["scale"])
    assert gdr.chunk_fwd_workspace_bytes(shape) == gdr.chunk_fwd_workspace_bytes(shape, segments=8)
    check(x)


def test_split_long_sequence_full_size_sampled():
    """The GDN-2 recipe at 65536 tokens with 4 heads (B * H = 4): the default
    path splits every sequence into runs; two heads against the oracle."""
    x = wl.config_inputs(5, H=4)
    o, hT = split_forward(x)
    torch.cuda.synchronize()
    for h in (0, 3):
        xs = select(x, batches=[0], heads=[h])
        ro, rh = oracle_forward(xs)
        assert rel_err(o[0:1, :, h:h + 1].float().cpu(), ro) <= BAR
        assert rel_err(hT[0:1, h:h + 1].cpu(), rh) <= BAR
    assert torch.isfinite(o).all()

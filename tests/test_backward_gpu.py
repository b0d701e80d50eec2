"""GPU parity of the chunkwise backward (gdr_chunk_bwd) against the float64
oracle's chunk backward (oracle/backward.py, itself pinned to autograd and to
finite differences).

Bar, per gradient tensor on the same seeded inputs (the oracle sees the
dtype-rounded inputs and dO): max|d| / max|ref| <= 1e-4 for fp32 inputs and
2e-2 for bf16 inputs, as for the forward; the arithmetic is fp32, the
per-chunk products of bf16 inputs on single tf32 products (worst measured
error over the flag sweep ~2.3e-3).
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_10_gb300 as gdr
from gated_delta_rule_10_gb300 import workloads as wl
from oracle import backward as obw
from tests.gdr_testutil import TOL, f64, rel_err, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "g", "beta", "lam", "b", "w")


def _cotangents(x, seed):
    B, T, H, dk = x["q"].shape
    dv = x["v"].shape[-1]
    gen = torch.Generator().manual_seed(seed)
    dO = torch.randn(B, T, H, dv, generator=gen).to(x["q"].dtype)
    dhT = torch.randn(B, H, dk, dv, generator=gen) * 0.1
    return dO, dhT


def _oracle(x, dO, dhT, b, h):
    sel = lambda t: None if t is None else f64(t[b, :, h])
    S0 = None if x["h0"] is None else f64(x["h0"][b, h])
    return obw.chunked_backward(*(sel(x[n]) for n in NAMES), S0=S0, scale=x["scale"],
                                flags=x["flags"], dO=sel(dO), dST=f64(dhT[b, h]), C=64)


def check(x, seed=0, seqs=None, tol=None):
    dO, dhT = _cotangents(x, seed)
    d = to_dev(x)
    grads = gdr.chunk_bwd(d["q"], d["k"], d["v"], d["g"], dO.cuda(), d["beta"], d["lam"], d["b"],
                          d["w"], d["h0"], dhT.cuda(), scale=x["scale"], flags=x["flags"])
    torch.cuda.synchronize()
    B, H = x["q"].shape[0], x["q"].shape[2]
    tol = tol or TOL[x["q"].dtype]
    worst = 0.0
    for b, h in (seqs or [(bb, hh) for bb in range(B) for hh in range(H)]):
        ref = _oracle(x, dO, dhT, b, h)
        for n in NAMES:
            if x[n] is None:
                continue
            got = grads[n][b, :, h].cpu()
            e = rel_err(got, ref[n])
            worst = max(worst, e)
            assert e <= tol, (n, b, h, e)
        e = rel_err(grads["h0"][b, h].cpu(), ref["S0"])
        assert e <= tol, ("h0", b, h, e)
    return worst


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("flags", range(16))
def test_backward_every_flag(flags, dtype):
    x = wl.make_inputs(flags, 2, 64 * 2 + 13, 2, 64, 64, dtype, seed=200 + flags, h0_std=0.05)
    check(x, seed=flags)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("variant", ["gdn", "qdelta", "kda", "gdn2"])
def test_backward_widths(variant, dk, dv):
    x = wl.make_inputs(variant, 1, 64 * 3 + 1, 2, dk, dv, torch.bfloat16, seed=dk + dv,
                       h0_std=0.05)
    check(x, seed=dk)


@pytest.mark.parametrize("T", [1, 63, 64, 65])
def test_backward_short_sequences(T):
    x = wl.make_inputs("gdn2", 2, T, 3, 64, 64, torch.float32, seed=T, h0_std=0.05)
    check(x, seed=T)


def test_backward_no_initial_state():
    x = wl.make_inputs("kda", 2, 100, 2, 64, 64, torch.float32, seed=4)
    assert x["h0"] is None
    check(x, seed=4)


def test_backward_gated_deltanet_workload_every_sequence():
    """The 4 x 4096 x 16 x 128 bf16 workload; every (batch, head) sequence's nine
    gradients against the oracle."""
    x = wl.config_inputs(2, gen_device="cuda")
    check(x, seed=5)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("flags", [0, 1, 8, 7, 15])
def test_backward_against_autograd(flags, dtype):
    """The GPU gradients straight against float64 autograd through the token
    recurrence (no chunk structure in the reference at all)."""
    x = wl.make_inputs(flags, 1, 64 * 2 + 5, 2, 64, 128, dtype, seed=400 + flags, h0_std=0.05)
    dO, dhT = _cotangents(x, 40 + flags)
    d = to_dev(x)
    grads = gdr.chunk_bwd(d["q"], d["k"], d["v"], d["g"], dO.cuda(), d["beta"], d["lam"], d["b"],
                          d["w"], d["h0"], dhT.cuda(), scale=x["scale"], flags=x["flags"])
    torch.cuda.synchronize()
    tol = TOL[dtype]
    for h in range(2):
        sel = lambda t: None if t is None else f64(t[0, :, h])
        ref = obw.grad_autograd(*(sel(x[n]) for n in NAMES), S0=f64(x["h0"][0, h]),
                                scale=x["scale"], flags=x["flags"], dO=sel(dO),
                                dST=f64(dhT[0, h]))
        for n in NAMES:
            if x[n] is None:
                continue
            e = rel_err(grads[n][0, :, h].cpu(), ref[n])
            assert e <= tol, (n, h, e)
        assert rel_err(grads["h0"][0, h].cpu(), ref["S0"]) <= tol


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("variant", ["gdn", "kda", "gdn2"])
def test_backward_decay_past_its_range_is_reported(variant, dtype):
    """A chunk whose running log-decay sum falls below -80 (per row for the
    scalar decay, per key channel otherwise) makes the backward's status
    GDR_ERR_RANGE, naming the first such sequence and its chunk."""
    B, T, H = 2, 64 * 3 + 7, 2
    x = wl.make_inputs(variant, B, T, H, 128, 128, dtype, seed=71, h0_std=0.02)
    if x["g"].dim() == 4:
        x["g"][1, 64:128, 0, 9] = -1.5       # sequence b=1, h=0, chunk 1: -96 on one channel
    else:
        x["g"][1, 64:128, 0] = -1.5
    dO, dhT = _cotangents(x, 7)
    d = to_dev(x)
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_bwd(d["q"], d["k"], d["v"], d["g"], dO.cuda(), d["beta"], d["lam"], d["b"],
                      d["w"], d["h0"], dhT.cuda(), scale=x["scale"], flags=x["flags"],
                      check=True)
    assert e.value.code == 6
    assert "sequence 2, chunk 1" in str(e.value)


@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_backward_decay_inside_its_range(variant):
    """Running sums down to about -74 within a chunk: no report, and the
    gradients keep the fp32 bar against the oracle."""
    x = wl.make_inputs(variant, 1, 64 * 2, 2, 128, 128, torch.float32, seed=72, h0_std=0.05)
    x["g"] = torch.full_like(x["g"], -1.15)   # -73.6 over a full chunk
    if x["g"].dim() == 4:
        x["g"][..., ::2] = -0.01
    dO, dhT = _cotangents(x, 8)
    d = to_dev(x)
    gdr.chunk_bwd(d["q"], d["k"], d["v"], d["g"], dO.cuda(), d["beta"], d["lam"], d["b"], d["w"],
                  d["h0"], dhT.cuda(), scale=x["scale"], flags=x["flags"], check=True)
    check(x, seed=8)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_backward_write_strength_per_value_channel(dk, dv, dtype):
    """GDR_BETA_CHANNEL (token-order backward): every gradient against float64
    autograd through the token recurrence, over several chunks with a ragged
    tail, from an initial state and with a final-state cotangent."""
    x = wl.make_inputs("vbeta", 2, 64 * 2 + 9, 2, dk, dv, dtype, seed=500 + dk + dv, h0_std=0.05)
    assert x["flags"] == gdr.BETA_CHANNEL and x["beta"].dim() == 4
    dO, dhT = _cotangents(x, 50 + dk)
    d = to_dev(x)
    grads = gdr.chunk_bwd(d["q"], d["k"], d["v"], d["g"], dO.cuda(), d["beta"], None, None, None,
                          d["h0"], dhT.cuda(), scale=x["scale"], flags=x["flags"], check=True)
    torch.cuda.synchronize()
    tol = TOL[dtype]
    for b in range(2):
        for h in range(2):
            sel = lambda t: None if t is None else f64(t[b, :, h])
            ref = obw.grad_autograd(*(sel(x[n]) for n in ("q", "k", "v", "g", "beta")),
                                    S0=f64(x["h0"][b, h]), scale=x["scale"], flags=x["flags"],
                                    dO=sel(dO), dST=f64(dhT[b, h]))
            for n in ("q", "k", "v", "g", "beta"):
                e = rel_err(grads[n][b, :, h].cpu(), ref[n])
                assert e <= tol, (n, b, h, e)
            assert rel_err(grads["h0"][b, h].cpu(), ref["S0"]) <= tol


def test_backward_write_strength_without_states():
    """No initial state and no final-state cotangent (both zero), one short chunk."""
    x = wl.make_inputs("vbeta", 1, 23, 3, 128, 128, torch.float32, seed=77, h0_std=None)
    dO, _ = _cotangents(x, 9)
    d = to_dev(x)
    grads = gdr.chunk_bwd(d["q"], d["k"], d["v"], d["g"], dO.cuda(), d["beta"], scale=x["scale"],
                          flags=x["flags"])
    torch.cuda.synchronize()
    for h in range(3):
        sel = lambda t: None if t is None else f64(t[0, :, h])
        ref = obw.grad_autograd(*(sel(x[n]) for n in ("q", "k", "v", "g", "beta")), S0=None,
                                scale=x["scale"], flags=x["flags"], dO=sel(dO), dST=None)
        for n in ("q", "k", "v", "g", "beta"):
            assert rel_err(grads[n][0, :, h].cpu(), ref[n]) <= TOL[torch.float32], n
        assert rel_err(grads["h0"][0, h].cpu(), ref["S0"]) <= TOL[torch.float32]


def _token_bwd_check(x, seed, seqs=None):
    dO, dhT = _cotangents(x, seed)
    d = to_dev(x)
    grads = gdr.token_bwd(d["q"], d["k"], d["v"], d["g"], dO.cuda(), d["beta"], d["lam"], d["b"],
                          d["w"], d["h0"], dhT.cuda(), scale=x["scale"], flags=x["flags"])
    torch.cuda.synchronize()
    B, H = x["q"].shape[0], x["q"].shape[2]
    tol = TOL[x["q"].dtype]
    for b, h in (seqs or [(bb, hh) for bb in range(B) for hh in range(H)]):
        sel = lambda t: None if t is None else f64(t[b, :, h])
        S0 = None if x["h0"] is None else f64(x["h0"][b, h])
        ref = obw.grad_autograd(*(sel(x[n]) for n in NAMES), S0=S0, scale=x["scale"],
                                flags=x["flags"], dO=sel(dO), dST=f64(dhT[b, h]))
        for n in NAMES:
            if x[n] is None:
                continue
            e = rel_err(grads[n][b, :, h].cpu(), ref[n])
            assert e <= tol, (n, b, h, e)
        assert rel_err(grads["h0"][b, h].cpu(), ref["S0"]) <= tol, ("h0", b, h)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("flags", range(17))
def test_token_backward_every_flag(flags, dtype):
    """gdr_token_bwd (the recurrence reversed token by token) against float64
    autograd, every flag combination (16: the per-value-channel write strength)."""
    x = wl.make_inputs(flags, 2, 64 * 2 + 9, 2, 128, 128, dtype, seed=700 + flags, h0_std=0.05)
    _token_bwd_check(x, 70 + flags)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("flags", [0, 7, 15])
def test_token_backward_widths(flags, dk, dv):
    x = wl.make_inputs(flags, 1, 64 + 23, 3, dk, dv, torch.float32, seed=800 + flags + dk + dv,
                       h0_std=0.05)
    _token_bwd_check(x, 90 + flags)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("variant", ["kda", "gdn2"])
def test_backward_channel_decay_minus_300_per_chunk(variant, dtype):
    """Per-channel in-chunk log-decay sums of -300: the chunk backward reports
    GDR_ERR_RANGE for them, and the token-order backward keeps the bar against
    float64 autograd."""
    x = wl.make_inputs(variant, 1, 64 * 2 + 5, 2, 128, 128, dtype, seed=41, h0_std=0.1)
    g = -300.0 / 64 * torch.ones_like(x["g"])
    g[..., 1::3] = -0.02                      # some channels keep their memory
    x["g"] = g.contiguous()
    dO, dhT = _cotangents(x, 42)
    d = to_dev(x)
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_bwd(d["q"], d["k"], d["v"], d["g"], dO.cuda(), d["beta"], d["lam"], d["b"],
                      d["w"], d["h0"], dhT.cuda(), scale=x["scale"], flags=x["flags"],
                      check=True)
    assert e.value.code == 6
    _token_bwd_check(x, 42)


@pytest.mark.parametrize("flags", [0, 7, 16])
def test_token_backward_single_token(flags):
    """T = 1: one chunk of one token (the checkpoint is the initial state)."""
    x = wl.make_inputs(flags, 2, 1, 2, 128, 128, torch.float32, seed=900 + flags, h0_std=0.05)
    _token_bwd_check(x, 95 + flags)

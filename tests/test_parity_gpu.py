"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Bar (element by element on the same seeded inputs): max|d| / max|ref| <= 1e-4
for fp32 inputs and <= 2e-2 for bf16 inputs, for both o and the final state.
Small cases compare every output; the full-size workloads run in the launch
configuration the benchmark times and compare every output too, the oracle
taking a few heads at a time so that host memory stays bounded.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_10_gb300 as gdr
from gated_delta_rule_10_gb300 import workloads as wl
from oracle import chunked as och
from tests.gdr_testutil import (TOL, ErrAcc, decode_as_sequences, f64,
                                full_parity, gpu_forward, oracle_forward, rel_err, select,
                                to_dev)

pytestmark = pytest.mark.gpu

VARIANTS = ["gdn", "qdelta", "kda", "gdn2"]
DTYPES = [torch.float32, torch.bfloat16]


def check(x, h0_std=None, tol=None, **kw):
    o, hT = gpu_forward(x, **kw)
    torch.cuda.synchronize()
    ro, rh = oracle_forward(x)
    tol = tol or TOL[x["q"].dtype]
    eo, eh = rel_err(o.float().cpu(), ro), rel_err(hT.cpu(), rh)
    assert eo <= tol and eh <= tol, (eo, eh)
    return eo, eh


@pytest.mark.parametrize("dtype", DTYPES, ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
@pytest.mark.parametrize("variant", VARIANTS)
def test_variants_small_shapes(variant, T, dk, dv, dtype):
    x = wl.make_inputs(variant, 2, T, 3, dk, dv, dtype, seed=T + dk + 7 * dv, h0_std=0.05)
    check(x)


@pytest.mark.parametrize("dtype", DTYPES, ids=["f32", "bf16"])
@pytest.mark.parametrize("flags", range(16))
def test_every_flag_combination(flags, dtype):
    x = wl.make_inputs(flags, 1, 130, 2, 128, 64, dtype, seed=100 + flags, h0_std=0.05)
    check(x)


# bf16 has two paths: the two-kernel one (full workspace, used above) and the
# single-kernel one (minimum workspace); both must meet the same bar.
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 65, 130])
@pytest.mark.parametrize("variant", VARIANTS)
def test_single_kernel_path_small_shapes(variant, T, dk, dv):
    x = wl.make_inputs(variant, 2, T, 3, dk, dv, torch.bfloat16, seed=T + dk + 7 * dv + 1,
                       h0_std=0.05)
    check(x, single_kernel=True)


@pytest.mark.parametrize("flags", range(16))
def test_single_kernel_path_every_flag_combination(flags):
    x = wl.make_inputs(flags, 1, 200, 2, 128, 128, torch.bfloat16, seed=300 + flags, h0_std=0.05)
    check(x, single_kernel=True)


@pytest.mark.parametrize("variant", VARIANTS)
def test_two_paths_agree(variant):
    """Same inputs through both bf16 paths: each within the bar of the other."""
    x = wl.make_inputs(variant, 2, 333, 4, 128, 128, torch.bfloat16, seed=77, h0_std=0.02)
    o1, h1 = gpu_forward(x)
    o2, h2 = gpu_forward(x, single_kernel=True)
    torch.cuda.synchronize()
    assert rel_err(o1.float().cpu(), o2.float().cpu().double().numpy()) <= TOL[torch.bfloat16]
    assert rel_err(h1.cpu(), h2.cpu().double().numpy()) <= TOL[torch.bfloat16]


def test_zero_initial_state_and_no_final_state():
    x = wl.make_inputs("kda", 1, 200, 2, 128, 128, torch.bfloat16, seed=5)
    o, hT = gpu_forward(x, output_final_state=False)
    assert hT is None
    ro, _ = oracle_forward(x)
    assert rel_err(o.float().cpu(), ro) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_workload_recipes_reduced_length(cfg):
    """Each named workload's recipe at a length the oracle finishes in seconds."""
    c = wl.CONFIGS[cfg]
    x = wl.config_inputs(cfg, T=min(c["T"], 320), B=min(c["B"], 2), H=min(c["H"], 4))
    check(x)


def test_config1_full_size():
    check(wl.config_inputs(1))


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_workload_full_size_every_sequence(cfg):
    """Full size, in the launch configuration the benchmark times (the library's
    recommended time segments, so the pipelined call for the Gated DeltaNet-2
    prefill); every element of o and hT of every (batch, head) against the
    oracle, streamed over groups of heads."""
    x = wl.config_inputs(cfg, gen_device="cuda")
    o, hT = gpu_forward(x, pipeline="auto")
    torch.cuda.synchronize()
    eo, eh = full_parity(x, o, hT)
    assert eo <= TOL[torch.bfloat16] and eh <= TOL[torch.bfloat16], (cfg, eo, eh)


@pytest.mark.parametrize("variant", ["gdn", "gdn2"])
def test_many_chunks_with_ragged_tail(variant):
    """More chunks than the persistent preparation grid holds at once (two CTAs
    per SM), a ragged last chunk, and both value slices of the scan; sampled
    (batch, head) pairs against the oracle."""
    B, H, T = 2, 6, 64 * 40 + 23          # 2 * 6 * 41 = 492 chunks
    x = wl.make_inputs(variant, B, T, H, 128, 128, torch.bfloat16, seed=55, h0_std=0.02)
    o, hT = gpu_forward(x)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (1, 5), (0, 3)]:
        xs = select(x, batches=[b], heads=[h])
        ro, rh = oracle_forward(xs)
        eo = rel_err(o[b:b + 1, :, h:h + 1].float().cpu(), ro)
        eh = rel_err(hT[b:b + 1, h:h + 1].cpu(), rh)
        assert eo <= TOL[torch.bfloat16] and eh <= TOL[torch.bfloat16], (b, h, eo, eh)


def test_scalar_decay_far_below_channel_limit():
    # scalar gates have no in-chunk range limit: sum over a chunk ~ -320
    x = wl.make_inputs("gdn", 1, 192, 2, 64, 64, torch.float32, seed=3, h0_std=0.1)
    x["g"] = torch.full_like(x["g"], -5.0)
    check(x)


def test_channel_decay_near_documented_limit():
    x = wl.make_inputs("kda", 1, 128, 2, 128, 128, torch.float32, seed=4, h0_std=0.1)
    x["g"] = torch.full_like(x["g"], -2.15)    # -137.6 over a full chunk
    x["g"][..., ::2] = -0.01
    check(x)


@pytest.mark.parametrize("variant", ["kda", "gdn2"])
def test_channel_decay_past_the_limit_is_reported(variant):
    """A chunk whose summed channel log-decay is below -140 makes the call's
    status GDR_ERR_RANGE (naming the sequence and chunk); chunks inside the
    limit (-137.6, the test above) report nothing."""
    B, T, H = 1, 200, 2
    x = wl.make_inputs(variant, B, T, H, 128, 128, torch.bfloat16, seed=14, h0_std=0.02)
    x["g"][0, 64:128, 1, 5] = -2.5          # chunk 1 of head 1: -160 on one channel
    with pytest.raises(gdr.GdrError) as e:
        gpu_forward(x)
    assert e.value.code == 6
    assert "sequence 1, chunk 1" in str(e.value)


def _token_forward(x):
    d = to_dev(x)
    return gdr.token_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"], d["b"], d["w"],
                         d["h0"], scale=x["scale"], flags=x["flags"])


@pytest.mark.parametrize("dtype", DTYPES, ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("flags", range(16))
def test_token_forward_every_flag(flags, dk, dv, dtype):
    """gdr_token_fwd (the recurrence token by token, fp32 state) against the oracle."""
    x = wl.make_inputs(flags, 2, 77, 3, dk, dv, dtype, seed=600 + flags, h0_std=0.05)
    o, hT = _token_forward(x)
    torch.cuda.synchronize()
    ro, rh = oracle_forward(x)
    tol = TOL[dtype]
    assert rel_err(o.float().cpu(), ro) <= tol and rel_err(hT.cpu(), rh) <= tol


@pytest.mark.parametrize("dtype", DTYPES, ids=["f32", "bf16"])
@pytest.mark.parametrize("variant", ["kda", "gdn2"])
def test_channel_decay_minus_300_per_chunk(variant, dtype):
    """Per-channel in-chunk log-decay sums of -300 (past the chunked path's
    range, which reports GDR_ERR_RANGE for them): the token-order path matches
    the oracle at the forward's bar, o and the final state."""
    x = wl.make_inputs(variant, 2, 200, 3, 128, 128, dtype, seed=31, h0_std=0.1)
    g = -300.0 / 64 * torch.ones_like(x["g"])
    g[..., 1::3] = -0.02                      # some channels keep their memory
    x["g"] = g.contiguous()
    if dtype == torch.bfloat16:
        with pytest.raises(gdr.GdrError) as e:
            gpu_forward(x)
        assert e.value.code == 6
    o, hT = _token_forward(x)
    torch.cuda.synchronize()
    ro, rh = oracle_forward(x)
    tol = TOL[dtype]
    assert rel_err(o.float().cpu(), ro) <= tol and rel_err(hT.cpu(), rh) <= tol


def test_token_forward_h0_and_hT_may_alias():
    x = wl.make_inputs("gdn2", 2, 90, 2, 128, 64, torch.float32, seed=32, h0_std=0.05)
    d = to_dev(x)
    state = d["h0"].clone()
    o, _ = gdr.token_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"], d["b"], d["w"],
                         state, hT=state, scale=x["scale"], flags=x["flags"])
    torch.cuda.synchronize()
    ro, rh = oracle_forward(x)
    assert rel_err(o.cpu(), ro) <= 1e-4 and rel_err(state.cpu(), rh) <= 1e-4


def test_unnormalised_keys_and_extended_erase_range():
    # b in [0, 2] (the extended erase range of the Gated DeltaNet-2 ablations)
    x = wl.make_inputs("gdn2", 1, 130, 2, 64, 64, torch.float32, seed=9, h0_std=0.1)
    x["b"] = 2.0 * x["b"]
    check(x)


def test_streaming_split_prefill_equals_whole():
    x = wl.make_inputs("qdelta", 2, 300, 3, 128, 128, torch.float32, seed=21, h0_std=0.05)
    o_full, h_full = gpu_forward(x)
    cut = 100   # not a chunk boundary
    p1 = {n: (t[:, :cut].contiguous() if torch.is_tensor(t) and n in
              ("q", "k", "v", "g", "beta", "lam", "b", "w") else t) for n, t in x.items()}
    p2 = {n: (t[:, cut:].contiguous() if torch.is_tensor(t) and n in
              ("q", "k", "v", "g", "beta", "lam", "b", "w") else t) for n, t in x.items()}
    o1, h1 = gpu_forward(p1)
    p2["h0"] = h1.cpu()
    o2, h2 = gpu_forward(p2)
    torch.cuda.synchronize()
    o_split = torch.cat([o1, o2], dim=1)
    assert rel_err(o_split.cpu(), o_full.cpu().numpy()) <= 1e-4
    assert rel_err(h2.cpu(), h_full.cpu().numpy()) <= 1e-4


def test_h0_and_hT_may_alias():
    x = wl.make_inputs("gdn", 2, 130, 2, 64, 128, torch.bfloat16, seed=31, h0_std=0.05)
    d = to_dev(x)
    state = d["h0"].clone()
    o, _ = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=state, hT=state,
                         scale=x["scale"], flags=x["flags"])
    torch.cuda.synchronize()
    ro, rh = oracle_forward(x)
    assert rel_err(o.float().cpu(), ro) <= 2e-2
    assert rel_err(state.cpu(), rh) <= 2e-2


def test_bitwise_deterministic():
    x = wl.make_inputs("gdn2", 1, 500, 4, 128, 128, torch.bfloat16, seed=41, h0_std=0.02)
    o1, h1 = gpu_forward(x)
    o2, h2 = gpu_forward(x)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_outputs_only_where_expected():
    # the kernel writes o only for the given tokens: a sentinel around it survives
    x = wl.make_inputs("gdn", 1, 70, 2, 64, 64, torch.bfloat16, seed=51)
    d = to_dev(x)
    buf = torch.full((2 * 70 * 2 * 64,), 7.0, dtype=torch.bfloat16, device="cuda")
    o = buf[:70 * 2 * 64].view(1, 70, 2, 64)
    gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"], o=o,
                  output_final_state=False)
    torch.cuda.synchronize()
    assert torch.all(buf[70 * 2 * 64:] == 7.0)


# ---------------------------------------------------------------- decode step
def _step_inputs(variant, N, H, dk, dv, dtype, seed):
    y = wl.make_inputs(variant, N, 1, H, dk, dv, dtype, seed=seed)
    return y


def _gpu_step(y, state):
    d = to_dev(y)
    sq = lambda t: None if t is None else t[:, 0].contiguous()
    return gdr.recurrent_step(sq(d["q"]), sq(d["k"]), sq(d["v"]), sq(d["g"]), state,
                              beta=sq(d["beta"]), lam=sq(d["lam"]), b=sq(d["b"]),
                              w=sq(d["w"]), scale=y["scale"], flags=y["flags"])


@pytest.mark.parametrize("dtype", DTYPES, ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("flags", range(16))
def test_recurrent_step_every_variant(flags, dk, dv, dtype):
    N, H, steps = 3, 2, 3
    gen = torch.Generator().manual_seed(flags)
    h0 = torch.randn(N, H, dk, dv, generator=gen) * 0.05
    state = h0.cuda()
    ys = [_step_inputs(flags, N, H, dk, dv, dtype, seed=1000 * flags + s) for s in range(steps)]
    outs = [_gpu_step(y, state) for y in ys]
    torch.cuda.synchronize()
    cat = {n: (torch.cat([y[n] for y in ys], dim=1) if ys[0][n] is not None else None)
           for n in ("q", "k", "v", "g", "beta", "lam", "b", "w")}
    cat.update(h0=h0, scale=ys[0]["scale"], flags=flags)
    ro, rh = oracle_forward(cat)
    got = torch.stack([o.float().cpu() for o in outs], dim=1)
    tol = TOL[dtype]
    assert rel_err(got, ro) <= tol and rel_err(state.cpu(), rh) <= tol


def test_decode_workload_every_step_and_sequence():
    """The Gated DeltaNet-2 decode phase as the benchmark runs it: 256 single-token
    steps at N=256, H=32, d=128 from random fp32 states, one gdr_recurrent_step
    call per token; every output of every step and the final state of every
    (sequence, head) against the oracle (each sequence's 256 tokens as one
    recurrence from its starting state)."""
    y = wl.decode_phase_inputs(5, gen_device="cuda")
    steps, N, H = y["q"].shape[:3]
    d = to_dev(y)
    state = d["h0"].clone()
    o = torch.empty(steps, N, H, y["v"].shape[-1], dtype=y["q"].dtype, device="cuda")
    g = lambda n, s: None if d[n] is None else d[n][s]
    for s in range(steps):
        gdr.recurrent_step(g("q", s), g("k", s), g("v", s), g("g", s), state, beta=g("beta", s),
                           lam=g("lam", s), b=g("b", s), w=g("w", s), scale=y["scale"],
                           flags=y["flags"], o=o[s])
    torch.cuda.synchronize()
    eo, eh = ErrAcc(), ErrAcc()
    for h0 in range(0, H, 4):
        hs = list(range(h0, h0 + 4))
        ro, rh = oracle_forward(decode_as_sequences(y, hs))
        eo.add(o[:, :, h0:h0 + 4].transpose(0, 1).float().cpu(), ro)
        eh.add(state[:, h0:h0 + 4].cpu(), rh)
    assert eo.value() <= TOL[torch.bfloat16] and eh.value() <= TOL[torch.bfloat16], (
        eo.value(), eh.value())


def test_prefill_then_decode_equals_longer_prefill():
    x = wl.make_inputs("kda", 2, 130, 2, 128, 128, torch.float32, seed=61, h0_std=0.05)
    o, hT = gpu_forward(x)
    y = wl.make_inputs("kda", 2, 1, 2, 128, 128, torch.float32, seed=62)
    o1 = _gpu_step(y, hT)
    torch.cuda.synchronize()
    cat = {n: (torch.cat([x[n], y[n]], dim=1) if x[n] is not None else None)
           for n in ("q", "k", "v", "g", "beta", "lam", "b", "w")}
    cat.update(h0=x["h0"], scale=x["scale"], flags=x["flags"])
    ro, rh = oracle_forward(cat)
    assert rel_err(o1.float().cpu(), ro[:, -1]) <= 1e-4
    assert rel_err(hT.cpu(), rh) <= 1e-4


# ------------------------------------------------------------ gate cumsum
@pytest.mark.parametrize("shape", [(2, 130, 3), (1, 200, 4, 128), (2, 64, 5, 64), (1, 1, 7)])
def test_gate_cumsum(shape):
    gen = torch.Generator().manual_seed(len(shape))
    g = -torch.nn.functional.softplus(torch.randn(*shape, generator=gen))
    G = gdr.gate_cumsum(g.cuda())
    torch.cuda.synchronize()
    ref = np.stack([och.chunk_local_cumsum(f64(g[b]), 64) for b in range(shape[0])])
    assert np.max(np.abs(G.cpu().numpy() - ref)) <= 1e-5 * max(1.0, np.abs(ref).max())


def test_gate_cumsum_in_place():
    g = -torch.rand(2, 100, 8, 64, device="cuda")
    ref = gdr.gate_cumsum(g.clone())
    gdr.gate_cumsum(g, out=g)
    torch.cuda.synchronize()
    assert torch.equal(g, ref)


# ------------------------------------------------------------ error paths
def test_binding_errors_on_gpu():
    x = to_dev(wl.make_inputs("gdn", 1, 64, 1, 64, 64, torch.bfloat16, seed=1))
    with pytest.raises(ValueError):
        gdr.chunk_fwd(x["q"], x["k"], x["v"].float(), x["g"], x["beta"])
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], None, flags=0)
    assert e.value.code == 1
    q = torch.zeros(1, 64, 1, 32, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_fwd(q, q, q, x["g"], x["beta"])
    assert e.value.code == 2


def test_many_sequences_few_chunks():
    """B * H = 768 sequences of three chunks: the persistent preparation grid walks
    2304 chunks in several passes and the scan runs 1536 CTAs; sampled sequences."""
    B, H, T = 24, 32, 64 * 2 + 9
    x = wl.make_inputs("kda", B, T, H, 64, 128, torch.bfloat16, seed=91, h0_std=0.02)
    o, hT = gpu_forward(x)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (23, 31), (11, 17)]:
        xs = select(x, batches=[b], heads=[h])
        ro, rh = oracle_forward(xs)
        eo = rel_err(o[b:b + 1, :, h:h + 1].float().cpu(), ro)
        eh = rel_err(hT[b:b + 1, h:h + 1].cpu(), rh)
        assert eo <= TOL[torch.bfloat16] and eh <= TOL[torch.bfloat16], (b, h, eo, eh)


def test_calls_on_two_streams():
    """Two forwards with their own workspaces on two streams at once agree with the
    oracle (nothing in the library is shared between calls)."""
    xs = [wl.make_inputs(v, 2, 300, 4, 128, 128, torch.bfloat16, seed=s, h0_std=0.02)
          for v, s in (("gdn", 1), ("gdn2", 2))]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for x, st in zip(xs, streams):
        d = to_dev(x)
        shape = gdr.make_shape(2, 300, 4, 128, 128, torch.bfloat16, x["flags"], x["scale"])
        ws = torch.empty(gdr.chunk_fwd_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            outs.append(gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"],
                                      d["b"], d["w"], d["h0"], scale=x["scale"],
                                      flags=x["flags"], workspace=ws, stream=st) + (ws, st))
    torch.cuda.synchronize()
    for x, (o, hT, ws, st) in zip(xs, outs):
        gdr.chunk_fwd_check(ws, stream=st)
        ro, rh = oracle_forward(x)
        assert rel_err(o.float().cpu(), ro) <= TOL[torch.bfloat16]
        assert rel_err(hT.cpu(), rh) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("N,H", [(1, 1), (153, 1), (19, 16)])
def test_recurrent_step_item_counts(N, H):
    """The decode stream with one item, with one item more than the SMs (one CTA
    takes two), and with several items per CTA: every output and state against
    the oracle over a few steps."""
    flags, dk, dv, dtype, steps = 7, 128, 128, torch.bfloat16, 3
    gen = torch.Generator().manual_seed(N * 31 + H)
    h0 = torch.randn(N, H, dk, dv, generator=gen) * 0.05
    state = h0.cuda()
    ys = [_step_inputs(flags, N, H, dk, dv, dtype, seed=5000 + 10 * N + s) for s in range(steps)]
    outs = [_gpu_step(y, state) for y in ys]
    torch.cuda.synchronize()
    cat = {n: (torch.cat([y[n] for y in ys], dim=1) if ys[0][n] is not None else None)
           for n in ("q", "k", "v", "g", "beta", "lam", "b", "w")}
    cat.update(h0=h0, scale=ys[0]["scale"], flags=flags)
    ro, rh = oracle_forward(cat)
    got = torch.stack([o.float().cpu() for o in outs], dim=1)
    tol = TOL[dtype]
    assert rel_err(got, ro) <= tol and rel_err(state.cpu(), rh) <= tol

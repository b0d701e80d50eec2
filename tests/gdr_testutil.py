"""Helpers shared by the GPU parity tests (not collected as tests).

Inputs come from ``gated_delta_rule_10_gb300.workloads`` (seeded, CPU); the
reference values from the float64 oracle (``oracle.native``), which sees the
same inputs after the dtype cast, upcast to fp64.
"""
import numpy as np
import torch

from oracle import native

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}   # max|d| / max|ref|
GATES = ("q", "k", "v", "g", "beta", "lam", "b", "w")


def to_dev(x, dev="cuda"):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}


def f64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def select(x, batches=None, heads=None):
    """The inputs restricted to some batch rows and heads (for sampled checks)."""
    out = dict(x)
    for n in GATES + ("h0",):
        t = x.get(n)
        if t is None:
            continue
        if batches is not None:
            t = t[batches]
        if heads is not None:
            t = t[:, heads] if n == "h0" else t[:, :, heads]
        out[n] = t.contiguous()
    return out


def oracle_forward(x, nthreads=0):
    """Float64 token recurrence of the whole input dict. Returns (o, hT)."""
    return native.recurrence(*(f64(x[n]) for n in ("q", "k", "v", "g")),
                             beta=f64(x["beta"]), lam=f64(x["lam"]), b=f64(x["b"]),
                             w=f64(x["w"]), h0=f64(x["h0"]), scale=x["scale"],
                             flags=x["flags"], nthreads=nthreads)


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output"
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


class ErrAcc:
    """max|got - ref| and max|ref| accumulated over pieces of one output, so that
    a full-size comparison can stream (batch, head) groups through the oracle and
    still report the same max|d| / max|ref| as one comparison of the whole."""

    def __init__(self):
        self.diff = 0.0
        self.ref = 0.0

    def add(self, got, ref):
        got = np.asarray(got, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        assert got.shape == ref.shape, (got.shape, ref.shape)
        assert np.all(np.isfinite(got)), "non-finite output"
        self.diff = max(self.diff, float(np.max(np.abs(got - ref))))
        self.ref = max(self.ref, float(np.max(np.abs(ref))))

    def value(self):
        return self.diff / max(self.ref, 1e-30)


def full_parity(x, o, hT, heads_per_group=8):
    """Every (batch, head) sequence of a forward's outputs o [B,T,H,d_v] and hT
    [B,H,d_k,d_v] (device tensors) against the oracle, streamed over groups of
    heads with all host cores busy inside each group. Returns the relative
    errors (o, hT) over the whole tensors."""
    B, T, H = x["q"].shape[:3]
    eo, eh = ErrAcc(), ErrAcc()
    for h0 in range(0, H, heads_per_group):
        hs = list(range(h0, min(H, h0 + heads_per_group)))
        ro, rh = oracle_forward(select(x, heads=hs))
        eo.add(o[:, :, hs[0]:hs[-1] + 1].float().cpu(), ro)
        del ro
        if hT is not None:
            eh.add(hT[:, hs[0]:hs[-1] + 1].cpu(), rh)
    return eo.value(), (eh.value() if hT is not None else 0.0)


def decode_as_sequences(y, heads):
    """Decode inputs [steps, N, H, d] as the oracle's [N, steps, H', d] sequences
    (sequence n, token s), restricted to some heads; h0 restricted alike."""
    out = dict(y)
    for n in GATES:
        t = y.get(n)
        if t is not None:
            out[n] = t[:, :, heads].transpose(0, 1).contiguous()
    out["h0"] = y["h0"][:, heads].contiguous()
    return out


def gpu_forward(x, single_kernel=False, pipeline=None, **kw):
    """The chunked forward through the C ABI; checks the call's status words.
    bf16 runs the two-kernel path, or with single_kernel=True the minimum
    workspace and so the single-kernel path. pipeline="auto" takes the time
    segments the library recommends for the shape (what the benchmark runs)."""
    import gated_delta_rule_10_gb300 as gdr
    d = to_dev(x)
    shape = gdr.make_shape(*d["q"].shape, d["v"].shape[-1], d["q"].dtype, x["flags"], x["scale"])
    if pipeline == "auto":
        pipeline = gdr.pipeline_segments(shape)
    if pipeline is not None and pipeline > 1:
        n = gdr.chunk_fwd_pipelined_workspace_bytes(shape, pipeline)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        out = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"], d["b"], d["w"],
                            d["h0"], scale=x["scale"], flags=x["flags"], workspace=ws,
                            pipeline=pipeline, **kw)
        gdr.chunk_fwd_check(ws)
        return out
    n = gdr.chunk_fwd_workspace_bytes(shape, minimum=single_kernel)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda") if (n or single_kernel) else None
    out = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"], d["b"], d["w"],
                        d["h0"], scale=x["scale"], flags=x["flags"], workspace=ws, **kw)
    gdr.chunk_fwd_check(ws)
    return out

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


def gpu_forward(x, single_kernel=False, **kw):
    """The chunked forward through the C ABI; checks the call's status words.
    bf16 runs the two-kernel path, or with single_kernel=True the minimum
    workspace and so the single-kernel path."""
    import gated_delta_rule_10_gb300 as gdr
    d = to_dev(x)
    shape = gdr.make_shape(*d["q"].shape, d["v"].shape[-1], d["q"].dtype, x["flags"], x["scale"])
    n = gdr.chunk_fwd_workspace_bytes(shape, minimum=single_kernel)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda") if (n or single_kernel) else None
    out = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["lam"], d["b"], d["w"],
                        d["h0"], scale=x["scale"], flags=x["flags"], workspace=ws, **kw)
    gdr.chunk_fwd_check(ws)
    return out

"""Seeded synthetic inputs for the gated delta rule (shared by tests and bench).

This module only draws random numbers and shapes them; it holds none of the
method's arithmetic, so both the CUDA path and the float64 oracle can take
their inputs from it without sharing any computation.

Recipe (one per variant, drawn in fp32 on the CPU with a seeded
``torch.Generator``, then cast to the compute dtype):

* q, k ~ N(0, 1), each token-head vector L2-normalised over its channels
  (the pages normalise q and k before the rule: Gated DeltaNet-2 notes,
  training strategy; LLMs from scratch ch. 11 section 11.3). With
  ``q_prescaled`` q is also multiplied by d_k^-1/2 and the read-out scale
  is 1, otherwise the read-out scale is d_k^-1/2.
* v ~ N(0, 1).
* scalar log-decay g = -softplus(N(0, 1)) per token and head (Gated
  DeltaNet, Q-Delta); channel log-decay g = -exp(N(-2, 0.5)) per key
  channel (KDA, Gated DeltaNet-2). Gates stay fp32.
* beta = sigmoid(N(0, 1)) per token and head; for the write strength per
  value channel (flag BETA_CHANNEL) beta = sigmoid(N(0, 1)) per token, head
  and value channel.
* Q-Delta: lambda ~ U[0, 1] per head, broadcast over batch and time; the
  write strength is capped so that beta * k^T x < 2 with x = k + lambda q:
  beta = sigmoid(N(0,1)) * min(1, 1.9 / (k^T x)) (factor 1 when k^T x <= 0),
  which keeps Q-Delta's one-step contraction condition (its notes, key
  design 4) true. k and q here are the values after the dtype cast.
* Gated DeltaNet-2: erase gate b = sigmoid(N(0, 1)) per key channel, write
  gate w = sigmoid(N(0, 1)) per value channel, in the compute dtype.
* Initial state (when asked for) ~ N(0, std^2) in fp32, layout
  [B, H, d_k, d_v].
* Output epilogue: read-out rows o ~ N(0, 0.05^2) (RMSNorm makes the scale
  immaterial), output-gate input z ~ N(0, 1), both in the compute dtype, and
  a near-unit gain weight = 1 + 0.1 N(0, 1) per value channel in fp32.

The five numbered workloads mirror the pages' 340M / 1.3B layer shapes; the
"vbeta" workload runs the per-value-channel write strength on workload 2's.
"""
import math

import torch

DECAY_CHANNEL = 1
ERASE_CHANNEL = 2
WRITE_CHANNEL = 4
QMIX = 8
BETA_CHANNEL = 16

VARIANT_FLAGS = {
    "gdn": 0,
    "qdelta": QMIX,
    "kda": DECAY_CHANNEL,
    "gdn2": DECAY_CHANNEL | ERASE_CHANNEL | WRITE_CHANNEL,
    "vbeta": BETA_CHANNEL,
}

# name -> recipe of the five workloads (the fifth also has a decode phase)
CONFIGS = {
    1: dict(name="gdn_fp32_b1_t256_h2_d64", variant="gdn", B=1, T=256, H=2, dk=64, dv=64,
            dtype=torch.float32, q_prescaled=True, h0_std=None, seed=0),
    2: dict(name="gdn_bf16_b4_t4096_h16_d128", variant="gdn", B=4, T=4096, H=16, dk=128,
            dv=128, dtype=torch.bfloat16, q_prescaled=False, h0_std=0.02, seed=1),
    3: dict(name="qdelta_bf16_b4_t8192_h16_d128", variant="qdelta", B=4, T=8192, H=16,
            dk=128, dv=128, dtype=torch.bfloat16, q_prescaled=False, h0_std=None, seed=2),
    4: dict(name="kda_bf16_b2_t16384_h32_d128", variant="kda", B=2, T=16384, H=32, dk=128,
            dv=128, dtype=torch.bfloat16, q_prescaled=False, h0_std=None, seed=3),
    5: dict(name="gdn2_bf16_b1_t65536_h32_d128", variant="gdn2", B=1, T=65536, H=32,
            dk=128, dv=128, dtype=torch.bfloat16, q_prescaled=False, h0_std=None, seed=4,
            decode=dict(steps=256, N=256, h_std=0.02)),
    # the write strength per value channel on workload 2's shapes
    "vbeta": dict(name="vbeta_bf16_b4_t4096_h16_d128", variant="vbeta", B=4, T=4096, H=16,
                  dk=128, dv=128, dtype=torch.bfloat16, q_prescaled=False, h0_std=0.02,
                  seed=6),
}


def _l2norm(x):
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def make_inputs(variant, B, T, H, dk, dv, dtype=torch.bfloat16, seed=0,
                q_prescaled=False, h0_std=None, device="cpu", gen_device=None):
    """Seeded inputs of one variant (a name or a flag bitmask), [B, T, H, d] layout.

    Returns a dict with q, k, v (dtype), g (fp32, [B,T,H] or [B,T,H,d_k]),
    beta / lam (fp32 [B,T,H] or None), b / w (dtype or None), h0 (fp32 or
    None), scale (float), flags (int) and variant.

    gen_device: where the numbers are drawn (default the CPU). The CPU
    generator is single-threaded, so the full-size workloads (a few hundred
    million values per tensor) are drawn on the GPU with a seeded CUDA
    generator instead: same recipe, different stream of numbers, and the
    tensors stay on that device. Whoever compares two paths hands both the
    same tensors.
    """
    if isinstance(variant, int):
        flags = variant                    # any flag combination, same recipe per gate
    elif variant in VARIANT_FLAGS:
        flags = VARIANT_FLAGS[variant]
    else:
        raise ValueError("unknown variant %r" % variant)
    gdev = torch.device(gen_device) if gen_device is not None else torch.device("cpu")
    gen = torch.Generator(device=gdev).manual_seed(int(seed))

    def normal(*shape, mean=0.0, std=1.0):
        return torch.randn(*shape, generator=gen, dtype=torch.float32, device=gdev) * std + mean

    q = _l2norm(normal(B, T, H, dk))
    k = _l2norm(normal(B, T, H, dk))
    if q_prescaled:
        q = q * dk ** -0.5
        scale = 1.0
    else:
        scale = dk ** -0.5
    v = normal(B, T, H, dv)
    q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)

    if flags & DECAY_CHANNEL:
        g = -torch.exp(normal(B, T, H, dk, mean=-2.0, std=0.5))
    else:
        g = -torch.nn.functional.softplus(normal(B, T, H))
    beta = lam = b = w = None
    if flags & BETA_CHANNEL:
        beta = torch.sigmoid(normal(B, T, H, dv))
    elif not (flags & ERASE_CHANNEL and flags & WRITE_CHANNEL):
        beta = torch.sigmoid(normal(B, T, H))
    if flags & QMIX:
        lam_h = torch.rand(H, generator=gen, dtype=torch.float32, device=gdev)
        lam = lam_h.view(1, 1, H).expand(B, T, H).contiguous()
    if flags & QMIX and beta is not None:
        kf, qf = k.float(), q.float()
        a = (kf * (kf + lam[..., None] * qf)).sum(-1)
        cap = torch.where(a > 0, torch.clamp(1.9 / a.clamp_min(1e-30), max=1.0),
                          torch.ones_like(a))
        beta = beta * cap
    if flags & ERASE_CHANNEL:
        b = torch.sigmoid(normal(B, T, H, dk)).to(dtype)
    if flags & WRITE_CHANNEL:
        w = torch.sigmoid(normal(B, T, H, dv)).to(dtype)
    h0 = None
    if h0_std is not None:
        h0 = normal(B, H, dk, dv, std=h0_std)
    out = dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta, lam=lam, b=b, w=w, h0=h0,
               scale=float(scale), flags=flags, variant=variant)
    if gen_device is None and torch.device(device) != gdev:
        out = {key: (val.to(device) if torch.is_tensor(val) else val) for key, val in out.items()}
    return out


def config_inputs(cfg_id, device="cpu", gen_device=None, **override):
    """Inputs of one of the five named workloads (prefill part); drawn on
    gen_device when given (and left there)."""
    c = dict(CONFIGS[cfg_id])
    c.update(override)
    return make_inputs(c["variant"], c["B"], c["T"], c["H"], c["dk"], c["dv"], c["dtype"],
                       c["seed"], c["q_prescaled"], c["h0_std"], device=device,
                       gen_device=gen_device)


def decode_phase_inputs(cfg_id=5, seed=None, gen_device=None, steps=None, **override):
    """The decode phase of a workload (the fifth has one): ``steps`` single-token
    steps for N sequences of H heads, as [steps, N, H, d] tensors (entry s is
    step s's contiguous [N, H, d] input, drawn with the prefill recipe), plus
    the starting states h0 [N, H, d_k, d_v] ~ N(0, h_std^2) fp32."""
    c = dict(CONFIGS[cfg_id])
    c.update(override)
    dec = c["decode"]
    steps = steps or dec["steps"]
    seed = c["seed"] + 500 if seed is None else seed
    y = make_inputs(c["variant"], steps, dec["N"], c["H"], c["dk"], c["dv"], c["dtype"],
                    seed=seed, gen_device=gen_device)
    gdev = torch.device(gen_device) if gen_device is not None else torch.device("cpu")
    gen = torch.Generator(device=gdev).manual_seed(int(seed) + 1)
    y["h0"] = torch.randn(dec["N"], c["H"], c["dk"], c["dv"], generator=gen,
                          device=gdev) * dec["h_std"]
    return y


def decode_inputs(variant, N, H, dk, dv, dtype=torch.bfloat16, seed=0, h_std=0.02,
                  device="cpu"):
    """One decode step's inputs: [N, 1, H, d] tensors plus a state [N, H, d_k, d_v]."""
    x = make_inputs(variant, N, 1, H, dk, dv, dtype, seed, False, h_std, device)
    return x


def epilogue_inputs(rows, dv, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Inputs of the output epilogue: o, z [rows, d_v] and weight [d_v], drawn
    on `device` with a generator seeded there."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(seed)
    o = (0.05 * torch.randn(rows, dv, generator=gen, device=dev)).to(dtype)
    z = torch.randn(rows, dv, generator=gen, device=dev).to(dtype)
    weight = 1.0 + 0.1 * torch.randn(dv, generator=gen, device=dev)
    return {"o": o, "z": z, "weight": weight}


def token_heads(cfg_id):
    c = CONFIGS[cfg_id]
    return c["B"] * c["T"] * c["H"]


def n_chunks(T, C=64):
    return math.ceil(T / C)

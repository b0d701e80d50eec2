"""Output epilogue of the gated delta rule block, float64 (oracle).

Test infrastructure only (see the package docstring).

The Gated DeltaNet-2 notes (overall framework, the last stage of its flow
chart) and the LLMs-from-scratch chapter 11 "Gated DeltaNet" (section 11.3,
the module's forward pass after the time loop) both follow the read-out o_t with RMSNorm and a SiLU output
gate before the heads are merged: the gate scales the representation already
read from the state and plays no part in writing it. Neither page spells the
formula out; the plain reading used here, per (token, head) row of d_v
channels, is

    y = o / sqrt(mean_c(o_c^2) + eps) * weight * silu(z),   silu(z) = z * sigmoid(z),

with `weight` the RMSNorm gain (one value per value channel, shared by the
heads) and `z` the gate input of the same shape as o.
"""
import numpy as np


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def rmsnorm_gate(o, z, weight, eps):
    """y = RMSNorm(o) * weight * silu(z) over the last axis, in float64."""
    o = np.asarray(o, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + float(eps))
    return o / rms * weight * silu(z)

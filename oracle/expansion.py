"""Closed-form product expansion of the gated delta rule, float64 (oracle).

Test infrastructure only (see the package docstring).

LLMs from scratch, ch. 11 "Gated DeltaNet", section 11.4: the recurrence
is affine, S_t = A_t S_{t-1} + U_t with A_t = alpha_t (I - beta_t k_t k_t^T)
and U_t = beta_t k_t v_t^T (state in d_k x d_v), so from the zero state
    S_t = sum_{i=1..t} (prod_{j=t..i+1} A_j) U_i,
the product applied right-to-left in time order. For the general variant
(Gated DeltaNet-2 notes, key design 1) the same holds with
A_t = (I - k_t e_t^T) D_t and U_t = k_t z_t^T. A nonzero initial state
adds (prod_{j=t..1} A_j) S_0. Section 11.6 reports this check on 6 tokens
of width 3 in float64 with a maximum error of 4.44e-16.
"""
import numpy as np

from .recurrence import erase_write_vectors, _f64


def transition_matrices(q, k, v, g, beta=None, lam=None, b=None, w=None, flags=0):
    """Per-token (A_t, U_t) of the affine form S_t = A_t S_{t-1} + U_t."""
    q, k, v, g = map(_f64, (q, k, v, g))
    T, dk = k.shape
    dv = v.shape[1]
    beta = np.zeros(T) if beta is None else _f64(beta)
    lam = np.zeros(T) if lam is None else _f64(lam)
    b = np.zeros((T, dk)) if b is None else _f64(b)
    w = np.zeros((T, dv)) if w is None else _f64(w)
    e, z = erase_write_vectors(q, k, v, beta, lam, b, w, flags)
    As, Us = [], []
    for t in range(T):
        alpha = np.exp(g[t]) * np.ones(dk)
        As.append((np.eye(dk) - np.outer(k[t], e[t])) @ np.diag(alpha))
        Us.append(np.outer(k[t], z[t]))
    return As, Us


def expanded_states(As, Us, S0=None):
    """All states S_1..S_T from the closed-form sum of products."""
    T = len(As)
    dk, dv = Us[0].shape
    states = []
    for t in range(T):                       # state after token t (0-based)
        S = np.zeros((dk, dv))
        for i in range(t + 1):
            P = np.eye(dk)
            for j in range(t, i, -1):        # A_t A_{t-1} ... A_{i+1}
                P = P @ As[j]
            S = S + P @ Us[i]
        if S0 is not None:
            P = np.eye(dk)
            for j in range(t, -1, -1):
                P = P @ As[j]
            S = S + P @ _f64(S0)
        states.append(S)
    return states

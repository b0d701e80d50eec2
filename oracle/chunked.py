"""Chunkwise WY/UT algebra of the gated delta rule, float64 (oracle).

Test infrastructure only (see the package docstring). This is the
algorithm of the Gated DeltaNet-2 notes, key design 2 ("absorbing the
cumulative decay into a chunkwise WY form"), taken step by step in the
notes' notation, for one sequence of one head, state S in R^{d_k x d_v}.
Q-Delta (key design 3 of its notes) reuses the same machinery with the
mixed input; scalar-gate Gated DeltaNet is the special case with alpha
broadcast over key channels.

Inside a chunk of C rows r = 1..C (the last chunk may be shorter):
    gamma_r   = exp(sum_{i<=r} g_i)                  per key channel
    k_bar_r   = gamma_r^{-1} (.) k_r,  e_bar_r = gamma_r (.) e_r
    T         = tril(E_bar K_bar^T, -1),  A = (I + T)^{-1}  (forward substitution)
    Y         = A E_bar,  U = A Z
    S_{n+1}   = Diag(gamma_C) S_n + K_tail^T (U - Y S_n)
    O_n       = Q_gamma S_n + A_qk (U - Y S_n)
The notes name K_tail, Q_gamma and A_qk without defining them. Writing
S_r = Diag(gamma_r) S^_r turns the recurrence into
S^_r = S^_{r-1} + k_bar_r u_r^T with u_r = z_r - S^_{r-1}^T e_bar_r, so
(I + T) U_true = Z - E_bar S_n, i.e. U_true = U - Y S_n, and then
    K_tail rows = gamma_C (.) gamma_r^{-1} (.) k_r
    Q_gamma rows = scale * gamma_r (.) q_r
    A_qk = tril(Q_gamma K_bar^T, 0)   (diagonal included: o_r reads the
                                       state after update r, ch. 11 s. 11.2)
"""
import numpy as np

from .recurrence import erase_write_vectors, _f64


def chunk_local_cumsum(g, C=64):
    """Inclusive prefix sum of the log-decay inside each chunk of C tokens.

    Gated DeltaNet-2 notes, key design 2 (gamma_r = exp(sum_{i<=r} g_i)
    restarts every chunk) and the training-strategy paragraph (the
    cumulative sum of g is taken in fp32 outside the kernel). Works on
    [T] or [T, d_k] arrays; chunks start at t = 0, C, 2C, ...
    """
    g = _f64(g)
    G = np.empty_like(g)
    for n0 in range(0, g.shape[0], C):
        acc = np.zeros(g.shape[1:])
        for t in range(n0, min(n0 + C, g.shape[0])):
            acc = acc + g[t]
            G[t] = acc
    return G


def forward_substitution_inverse(T):
    """A = (I + T)^{-1} for strictly lower-triangular T, row by row.

    Gated DeltaNet-2 notes, key design 2 ("reduced to a forward
    substitution"): row r of (I + T) A = I gives
    A_r = e_r - sum_{i<r} T_{r,i} A_i.
    """
    n = T.shape[0]
    A = np.zeros((n, n))
    for r in range(n):
        row = np.zeros(n)
        row[r] = 1.0
        for i in range(r):
            row -= T[r, i] * A[i]
        A[r] = row
    return A


def chunked(q, k, v, g, beta=None, lam=None, b=None, w=None, S0=None,
            scale=1.0, flags=0, C=64):
    """Chunkwise forward of one sequence; returns (o [T, d_v], S_T).

    Arguments as ``recurrence.unified``; g is [T] (scalar decay, broadcast
    over key channels) or [T, d_k].
    """
    q, k, v, g = map(_f64, (q, k, v, g))
    Tn, dk = k.shape
    dv = v.shape[1]
    beta = np.zeros(Tn) if beta is None else _f64(beta)
    lam = np.zeros(Tn) if lam is None else _f64(lam)
    b = np.zeros((Tn, dk)) if b is None else _f64(b)
    w = np.zeros((Tn, dv)) if w is None else _f64(w)
    E, Z = erase_write_vectors(q, k, v, beta, lam, b, w, flags)
    gk = g if g.ndim == 2 else np.repeat(g[:, None], dk, axis=1)
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    O = np.zeros((Tn, dv))
    for n0 in range(0, Tn, C):
        sl = slice(n0, min(n0 + C, Tn))
        gamma = np.exp(chunk_local_cumsum(gk[sl], C))      # [L, d_k]
        K_bar = k[sl] / gamma
        E_bar = gamma * E[sl]
        Tm = np.tril(E_bar @ K_bar.T, -1)
        A = forward_substitution_inverse(Tm)
        Y = A @ E_bar
        U = A @ Z[sl]
        gamma_C = gamma[-1]
        K_tail = (gamma_C / gamma) * k[sl]
        Q_gamma = scale * gamma * q[sl]
        A_qk = np.tril(Q_gamma @ K_bar.T, 0)
        W = U - Y @ S
        O[sl] = Q_gamma @ S + A_qk @ W
        S = gamma_C[:, None] * S + K_tail.T @ W
    return O, S

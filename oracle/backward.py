"""Gradients of the gated delta rule, float64 (oracle).

Test infrastructure only (see the package docstring). Two forms, one
sequence of one head at a time, loss L = <dO, O> + <dS_T, S_T>:

* ``grad_autograd`` -- PyTorch float64 autograd through the token recurrence
  of ``recurrence.unified`` (every flag, BETA_CHANNEL included): the gradient
  of the defined function, with the differentiation left to the library.
* ``chunked_backward`` -- the chunkwise backward of the Gated DeltaNet-2 notes,
  key design 3: the reverse state pass over chunks, the gate-aware
  accumulation dA += dU Z^T, dA += dY E_bar^T (the gates stay inside the
  products instead of being pulled out as scalars), the adjoint of the
  lower-triangular inverse dT = -tril(A^T dA A^T, -1), then the chain through
  the decay factors to g, b, w, beta and lam. The notes give those two
  formulas; every other line is the adjoint of one line of
  ``chunked.chunked``'s forward, in reverse order, and the pins check the whole
  against ``grad_autograd`` and against finite differences.
"""
import numpy as np
import torch

from .chunked import chunk_local_cumsum, forward_substitution_inverse
from .recurrence import BETA_CHANNEL, DECAY_CHANNEL, ERASE_CHANNEL, QMIX, WRITE_CHANNEL, _f64

NAMES = ("q", "k", "v", "g", "beta", "lam", "b", "w", "S0")


def _recurrence_torch(q, k, v, g, beta, lam, b, w, S0, scale, flags):
    """``recurrence.unified`` in PyTorch float64 ops, for autograd."""
    T = k.shape[0]
    S = S0
    outs = []
    for t in range(T):
        alpha = torch.exp(g[t])
        S_tilde = (alpha[:, None] if alpha.dim() else alpha) * S
        if flags & BETA_CHANNEL:
            e, z = k[t], v[t]
        else:
            x = k[t] + lam[t] * q[t] if flags & QMIX else k[t]
            e = b[t] * x if flags & ERASE_CHANNEL else beta[t] * x
            z = w[t] * v[t] if flags & WRITE_CHANNEL else beta[t] * v[t]
        err = z - S_tilde.T @ e
        if flags & BETA_CHANNEL:
            err = beta[t] * err
        S = S_tilde + torch.outer(k[t], err)
        outs.append(S.T @ (scale * q[t]))
    return torch.stack(outs), S


def grad_autograd(q, k, v, g, beta=None, lam=None, b=None, w=None, S0=None, scale=1.0,
                  flags=0, dO=None, dST=None):
    """Gradients of <dO, O> + <dS_T, S_T> by float64 autograd.

    Shapes as ``recurrence.unified``; beta is [T] or [T, d_v] (BETA_CHANNEL).
    Returns a dict over NAMES (None for an input that was not given; S0
    defaults to zeros and its gradient is always returned).
    """
    T, dk = np.shape(k)
    dv = np.shape(v)[1]
    vals = {"q": q, "k": k, "v": v, "g": g, "beta": beta, "lam": lam, "b": b, "w": w,
            "S0": np.zeros((dk, dv)) if S0 is None else S0}
    ts = {n: (None if a is None else torch.tensor(_f64(a), requires_grad=True))
          for n, a in vals.items()}
    zero = torch.zeros(T, dtype=torch.float64)
    args = [ts[n] if ts[n] is not None else (zero if n in ("beta", "lam") else
                                             torch.zeros(T, dk if n == "b" else dv,
                                                         dtype=torch.float64))
            for n in NAMES]
    O, ST = _recurrence_torch(*args, scale, flags)
    loss = (torch.tensor(_f64(dO)) * O).sum()
    if dST is not None:
        loss = loss + (torch.tensor(_f64(dST)) * ST).sum()
    live = [n for n in NAMES if ts[n] is not None]
    grads = torch.autograd.grad(loss, [ts[n] for n in live], allow_unused=True)
    out = {n: None for n in NAMES}
    for n, gr in zip(live, grads):
        out[n] = np.zeros(np.shape(vals[n])) if gr is None else gr.numpy()
    return out


def gate_aware_dA(dU, Z, dY, E_bar):
    """dA of Y = A E_bar, U = A Z (Gated DeltaNet-2 notes, key design 3): the
    per-row, per-channel gates stay inside the products, dA = dU Z^T + dY E_bar^T."""
    return dU @ Z.T + dY @ E_bar.T


def inverse_adjoint(A, dA):
    """dT of A = (I + T)^{-1} with T strictly lower (the notes' adjoint of the
    lower-triangular inverse): dT = -tril(A^T dA A^T, -1)."""
    return -np.tril(A.T @ dA @ A.T, -1)


def chunked_backward(q, k, v, g, beta=None, lam=None, b=None, w=None, S0=None, scale=1.0,
                     flags=0, dO=None, dST=None, C=64):
    """The chunkwise backward (Gated DeltaNet-2 notes, key design 3) of
    ``chunked.chunked`` for flags without BETA_CHANNEL. Same arguments and return
    as ``grad_autograd``."""
    assert not flags & BETA_CHANNEL, "the shared-inverse chunk form has no per-column beta"
    q, k, v, g = map(_f64, (q, k, v, g))
    Tn, dk = k.shape
    dv = v.shape[1]
    beta_ = np.zeros(Tn) if beta is None else _f64(beta)
    lam_ = np.zeros(Tn) if lam is None else _f64(lam)
    b_ = np.zeros((Tn, dk)) if b is None else _f64(b)
    w_ = np.zeros((Tn, dv)) if w is None else _f64(w)
    S0_ = np.zeros((dk, dv)) if S0 is None else _f64(S0)
    dO = _f64(dO)
    # erase input and vectors, as the forward forms them (recurrence.erase_write_vectors)
    x = k + lam_[:, None] * q if flags & QMIX else k
    E = b_ * x if flags & ERASE_CHANNEL else beta_[:, None] * x
    Z = w_ * v if flags & WRITE_CHANNEL else beta_[:, None] * v
    gk = g if g.ndim == 2 else np.repeat(g[:, None], dk, axis=1)

    # forward pass over the chunks, keeping the state entering each chunk
    chunks = [slice(n0, min(n0 + C, Tn)) for n0 in range(0, Tn, C)]
    states = []
    S = S0_.copy()
    cache = []
    for sl in chunks:
        gamma = np.exp(chunk_local_cumsum(gk[sl], C))
        K_bar = k[sl] / gamma
        E_bar = gamma * E[sl]
        A = forward_substitution_inverse(np.tril(E_bar @ K_bar.T, -1))
        Y, U = A @ E_bar, A @ Z[sl]
        gamma_C = gamma[-1]
        K_tail = (gamma_C / gamma) * k[sl]
        Q_gamma = scale * gamma * q[sl]
        A_qk = np.tril(Q_gamma @ K_bar.T, 0)
        states.append(S)
        W = U - Y @ S
        cache.append((gamma, K_bar, E_bar, A, Y, U, gamma_C, K_tail, Q_gamma, A_qk, W))
        S = gamma_C[:, None] * S + K_tail.T @ W

    dq, dk_, dv_ = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dE, dZ = np.zeros_like(E), np.zeros_like(Z)
    dg = np.zeros_like(gk)
    dS = np.zeros((dk, dv)) if dST is None else _f64(dST).copy()
    for sl, S_n, (gamma, K_bar, E_bar, A, Y, U, gamma_C, K_tail, Q_gamma, A_qk, W) in zip(
            reversed(chunks), reversed(states), reversed(cache)):
        dOn = dO[sl]
        # O = Q_gamma S_n + A_qk W,  S' = Diag(gamma_C) S_n + K_tail^T W
        dW = A_qk.T @ dOn + K_tail @ dS
        dA_qk = np.tril(dOn @ W.T, 0)
        dQ_gamma = dOn @ S_n.T + dA_qk @ K_bar
        dK_bar = dA_qk.T @ Q_gamma
        dK_tail = W @ dS.T
        dgamma_C = (dS * S_n).sum(axis=1)
        dS_prev = gamma_C[:, None] * dS + Q_gamma.T @ dOn
        # W = U - Y S_n
        dU = dW
        dY = -dW @ S_n.T
        dS_prev = dS_prev - Y.T @ dW
        # Y = A E_bar, U = A Z: the gate-aware accumulation of the notes
        dA = gate_aware_dA(dU, Z[sl], dY, E_bar)
        dZ[sl] += A.T @ dU
        dE_bar = A.T @ dY
        # A = (I + T)^{-1}, T = tril(E_bar K_bar^T, -1)
        dT = inverse_adjoint(A, dA)
        dE_bar += dT @ K_bar
        dK_bar += dT.T @ E_bar
        # the decay factors: K_bar = k / gamma, E_bar = gamma e,
        # K_tail = (gamma_C / gamma) k, Q_gamma = scale gamma q
        kk = k[sl]
        dk_[sl] += dK_bar / gamma + (gamma_C / gamma) * dK_tail
        dE[sl] += gamma * dE_bar
        dq[sl] += scale * gamma * dQ_gamma
        dgamma = (dE_bar * E[sl] - dK_bar * K_bar / gamma - dK_tail * K_tail / gamma
                  + dQ_gamma * Q_gamma / gamma)
        dgamma_C = dgamma_C + (dK_tail * kk / gamma).sum(axis=0)
        # gamma_r = exp(G_r), gamma_C = gamma of the chunk's last row, G = cumsum g
        dG = gamma * dgamma
        dG[-1] += gamma_C * dgamma_C
        dg[sl] += np.cumsum(dG[::-1], axis=0)[::-1]
        dS = dS_prev

    # e and z back to their inputs
    dx = b_ * dE if flags & ERASE_CHANNEL else beta_[:, None] * dE
    out = {n: None for n in NAMES}
    dbeta = np.zeros(Tn)
    if flags & ERASE_CHANNEL:
        out["b"] = x * dE
    else:
        dbeta += (x * dE).sum(axis=1)
    dk_ += dx
    if flags & QMIX:
        dq += lam_[:, None] * dx
        out["lam"] = (q * dx).sum(axis=1)
    if flags & WRITE_CHANNEL:
        dv_ += w_ * dZ
        out["w"] = v * dZ
    else:
        dv_ += beta_[:, None] * dZ
        dbeta += (v * dZ).sum(axis=1)
    if beta is not None:
        out["beta"] = dbeta
    out.update(q=dq, k=dk_, v=dv_, g=dg if g.ndim == 2 else dg.sum(axis=1), S0=dS)
    return out

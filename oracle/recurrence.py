"""Token-by-token recurrences of the gated delta rule, float64 (oracle).

Test infrastructure only (see the package docstring). Each function
handles ONE sequence of one head and is written from one page, in that
page's own orientation of the state, so that the reductions between them
(tests/test_oracle_pins.py) cross-check the orientations:

* ``gdn_llms_ch11``   -- state S in R^{d_k x d_v}
  (LLMs from scratch, ch. 11 "Gated DeltaNet", section 11.2).
* ``kda_kimi``        -- state S in R^{d_v x d_k}
  ("You could have come up with Kimi Delta Attention", section 4).
* ``gdn2_decoupled``  -- state S in R^{d_k x d_v}
  (Gated DeltaNet-2 notes, key design 1, the Gated Delta Rule-2 update).
* ``qdelta_q_delta_page`` -- state S in R^{d_v x d_k}
  (Q-Delta notes, key design 3, the rewritten rule with x_t = k_t + lam_t q_t).
* ``unified``         -- the one form the CUDA path implements, in the
  d_k x d_v orientation, with the variant chosen by flags.

Array conventions (one sequence): q, k: [T, d_k]; v: [T, d_v];
alpha or g: [T] (scalar gate) or [T, d_k] (per-channel gate);
beta, lam: [T]; b: [T, d_k]; w: [T, d_v]. Everything is float64.
"""
import numpy as np

# Variant flags. The numeric values mirror the C interface's bitmask so
# the tests can pass one integer to both sides; nothing here reads the
# product's headers.
DECAY_CHANNEL = 1   # g / alpha per key channel (KDA, GDN-2)
ERASE_CHANNEL = 2   # erase direction e_t = b_t (.) x_t   (GDN-2)
WRITE_CHANNEL = 4   # write vector   z_t = w_t (.) v_t   (GDN-2)
QMIX = 8            # erase input x_t = k_t + lam_t q_t  (Q-Delta)
BETA_CHANNEL = 16   # beta_t per value channel, scaling the error (ch. 11 README)


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def gdn_llms_ch11(q, k, v, alpha, beta, S0=None, scale=1.0):
    """Gated DeltaNet with scalar alpha_t, beta_t; S in R^{d_k x d_v}.

    LLMs from scratch, ch. 11 "Gated DeltaNet", section 11.2: decay the old
    state first (S~ = alpha_t S_{t-1}), predict from the decayed state
    (v^_t = S~^T k_t), write the beta-scaled error along k_t
    (S_t = S~ + beta_t k_t (v_t - v^_t)^T), read y_t = S_t^T q_t.
    Section 11.3 stresses that the decay comes before the prediction.
    ``scale`` multiplies q at read-out (1 reproduces the page exactly).
    """
    q, k, v, alpha, beta = map(_f64, (q, k, v, alpha, beta))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((T, dv))
    for t in range(T):
        S_tilde = alpha[t] * S
        v_hat = S_tilde.T @ k[t]
        S = S_tilde + beta[t] * np.outer(k[t], v[t] - v_hat)
        o[t] = S.T @ (scale * q[t])
    return o, S


def gdn_value_beta_ch11(q, k, v, alpha, beta_v, S0=None, scale=1.0):
    """Gated DeltaNet with a write strength per value channel; S in R^{d_k x d_v}.

    LLMs from scratch, ch. 11 "Gated DeltaNet", section 11.3: the chapter's
    README module draws its write gate per value channel and scales the
    prediction error channel by channel, while the forget gate stays one
    scalar per head; the decay comes before the prediction. So with
    beta_v in R^{d_v}: S~ = alpha_t S_{t-1}, v^_t = S~^T k_t,
    S_t = S~ + k_t (beta_v,t (.) (v_t - v^_t))^T, y_t = S_t^T q_t.
    Section 11.4 adds that each column of the state then follows its own
    affine update, which the pins use.
    """
    q, k, v, alpha, beta_v = map(_f64, (q, k, v, alpha, beta_v))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((T, dv))
    for t in range(T):
        S_tilde = alpha[t] * S
        v_hat = S_tilde.T @ k[t]
        S = S_tilde + np.outer(k[t], beta_v[t] * (v[t] - v_hat))
        o[t] = S.T @ (scale * q[t])
    return o, S


def kda_kimi(q, k, v, alpha, beta, S0_vk=None, scale=1.0):
    """Kimi Delta Attention; S in R^{d_v x d_k} (keys map to values).

    "You could have come up with Kimi Delta Attention", section 4: forget
    each key channel (S~ = S_{t-1} Diag(alpha_t), i.e. scale S's columns),
    predict v^_t = S~ k_t, correct e_t = beta_t (v_t - v^_t), write
    S_t = S~ + e_t k_t^T and read o_t = S_t (s q_t).
    ``alpha`` is [T, d_k]; the returned state keeps the page's d_v x d_k
    orientation (the caller transposes to compare).
    """
    q, k, v, alpha, beta = map(_f64, (q, k, v, alpha, beta))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0_vk is None else _f64(S0_vk).copy()
    o = np.zeros((T, dv))
    for t in range(T):
        S_tilde = S @ np.diag(alpha[t])
        v_hat = S_tilde @ k[t]
        e = beta[t] * (v[t] - v_hat)
        S = S_tilde + np.outer(e, k[t])
        o[t] = S @ (scale * q[t])
    return o, S


def gdn2_decoupled(q, k, v, alpha, b, w, S0=None, scale=1.0):
    """Gated DeltaNet-2; S in R^{d_k x d_v}.

    Gated DeltaNet-2 notes, key design 1 (the Gated Delta Rule-2 update):
    S_t = (I - k_t (b_t (.) k_t)^T) D_t S_{t-1} + k_t (w_t (.) v_t)^T with
    D_t = Diag(alpha_t), alpha_t in (0,1)^{d_k}, erase gate b_t over key
    channels and write gate w_t over value channels. Read-out follows the
    chunk output O = Q_gamma S + ... of key design 2, i.e. o_t = S_t^T q_t.
    """
    q, k, v, alpha, b, w = map(_f64, (q, k, v, alpha, b, w))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((T, dv))
    eye = np.eye(dk)
    for t in range(T):
        D = np.diag(alpha[t])
        S = (eye - np.outer(k[t], b[t] * k[t])) @ D @ S + np.outer(k[t], w[t] * v[t])
        o[t] = S.T @ (scale * q[t])
    return o, S


def qdelta_q_delta_page(q, k, v, alpha, beta, lam, S0_vk=None, scale=1.0):
    """Q-Delta; S in R^{d_v x d_k}.

    Q-Delta notes, key design 3: with the mixed input x_t = k_t + lam_t q_t
    the rule reads S_t = alpha_t S_{t-1} (I - beta_t x_t k_t^T)
    + beta_t v_t k_t^T, read out as o_t = S_t q_t (the notes' linear-attention
    read-out, research background).

    Parity unpinned on one point: the notes lost the display equations of
    key design 2, so which query enters x_t is a reading. Here it is the
    same (unscaled) q_t that is read out; ``scale`` only multiplies the
    read-out.
    """
    q, k, v, alpha, beta, lam = map(_f64, (q, k, v, alpha, beta, lam))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0_vk is None else _f64(S0_vk).copy()
    o = np.zeros((T, dv))
    eye = np.eye(dk)
    for t in range(T):
        x = k[t] + lam[t] * q[t]
        S = alpha[t] * S @ (eye - beta[t] * np.outer(x, k[t])) + beta[t] * np.outer(v[t], k[t])
        o[t] = S @ (scale * q[t])
    return o, S


def erase_write_vectors(q, k, v, beta, lam, b, w, flags):
    """Per-token erase direction e_t and write vector z_t of each variant.

    Gated DeltaNet (ch. 11 section 11.2) and KDA (section 4): e = beta k,
    z = beta v. Gated DeltaNet-2 (key design 1): e = b (.) k, z = w (.) v.
    Q-Delta (key design 3): the erase input becomes x = k + lam q, so
    e = beta x, z = beta v. Flags combine independently (the GDN-2
    ablation table uses channel b with scalar w and the reverse):
    x = k + lam q if QMIX else k; e = b (.) x if ERASE_CHANNEL else beta x;
    z = w (.) v if WRITE_CHANNEL else beta v.
    Under BETA_CHANNEL (ch. 11 section 11.3's README variant) beta is
    [T, d_v] and scales the error per value channel instead; the vectors
    returned are then the unscaled e = k and z = v, and ``unified`` applies
    beta to z - r.
    """
    if flags & BETA_CHANNEL:
        return k, v
    x = k + lam[:, None] * q if flags & QMIX else k
    e = b * x if flags & ERASE_CHANNEL else beta[:, None] * x
    z = w * v if flags & WRITE_CHANNEL else beta[:, None] * v
    return e, z


def unified(q, k, v, g, beta=None, lam=None, b=None, w=None, S0=None,
            scale=1.0, flags=0):
    """The form shared by all four variants; S in R^{d_k x d_v}.

    For t = 1..T (Gated DeltaNet-2 notes, key design 1, with e_t and z_t
    named there; order forget -> predict -> correct -> write -> read as the
    KDA derivation, section 3, insists):
        alpha_t = exp(g_t)                   (scalar or per key channel)
        S~      = Diag(alpha_t) S_{t-1}
        r_t     = S~^T e_t
        S_t     = S~ + k_t (z_t - r_t)^T
        o_t     = S_t^T (scale q_t)
    g is the log-decay; g = -inf gives alpha = 0 exactly. Under
    BETA_CHANNEL (README variant of ch. 11 section 11.3) beta is [T, d_v],
    e_t = k_t, z_t = v_t and the write becomes
        S_t     = S~ + k_t (beta_t (.) (v_t - r_t))^T.
    Returns (o [T, d_v], S_T [d_k, d_v]).
    """
    q, k, v, g = map(_f64, (q, k, v, g))
    T, dk = k.shape
    dv = v.shape[1]
    beta = np.zeros(T) if beta is None else _f64(beta)
    lam = np.zeros(T) if lam is None else _f64(lam)
    b = np.zeros((T, dk)) if b is None else _f64(b)
    w = np.zeros((T, dv)) if w is None else _f64(w)
    e, z = erase_write_vectors(q, k, v, beta, lam, b, w, flags)
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((T, dv))
    for t in range(T):
        alpha = np.exp(g[t])
        S_tilde = (alpha[:, None] if np.ndim(alpha) else alpha) * S
        r = S_tilde.T @ e[t]
        err = z[t] - r
        if flags & BETA_CHANNEL:
            err = beta[t] * err
        S = S_tilde + np.outer(k[t], err)
        o[t] = S.T @ (scale * q[t])
    return o, S


def unified_batched(q, k, v, g, beta=None, lam=None, b=None, w=None, h0=None,
                    scale=1.0, flags=0):
    """``unified`` over every (batch, head) of [B, T, H, d] arrays.

    Returns o [B, T, H, d_v] and the final states [B, H, d_k, d_v].
    """
    B, T, H, dk = np.shape(k)
    dv = np.shape(v)[-1]
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    for bi in range(B):
        for h in range(H):
            sel = lambda a: None if a is None else np.asarray(a)[bi, :, h]
            S0 = None if h0 is None else np.asarray(h0)[bi, h]
            o[bi, :, h], hT[bi, h] = unified(
                sel(q), sel(k), sel(v), sel(g), sel(beta), sel(lam), sel(b), sel(w),
                S0, scale, flags)
    return o, hT

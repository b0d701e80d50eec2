"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these compare the oracle with itself: each uses a value the pages
print, an identity they state, a closed form computed another way, or a
different page's formulation in another state orientation. Most cases use
d_k != d_v so a transposed operand fails on shape or on value.
"""
import json
import os

import numpy as np
import pytest

from oracle import chunked as ch
from oracle import expansion as ex
from oracle import native
from oracle import recurrence as rc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALL_FLAGS = list(range(16))


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def seq(rng, T, dk, dv, channel=False, s0=True):
    """A random sequence with the pages' gate ranges (fp64)."""
    d = dict(
        q=_unit(rng.standard_normal((T, dk))),
        k=_unit(rng.standard_normal((T, dk))),
        v=rng.standard_normal((T, dv)),
        g=-np.log1p(np.exp(rng.standard_normal((T, dk) if channel else T))),
        beta=_sig(rng.standard_normal(T)),
        lam=rng.uniform(size=T),
        b=_sig(rng.standard_normal((T, dk))),
        w=_sig(rng.standard_normal((T, dv))),
        S0=0.3 * rng.standard_normal((dk, dv)) if s0 else None,
    )
    return d


def relerr(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# --------------------------------------------------------------------------
# LLMs from scratch ch. 11, section 11.2: the worked example and key scaling
# --------------------------------------------------------------------------
def test_worked_example_row_overwrite():
    d = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    S_old = np.array(d["S_old"])
    k = np.array([d["k"]])
    v = np.array([d["v"]])
    q = k.copy()  # read back along the key just written
    o, S = rc.gdn_llms_ch11(q, k, v, np.array([d["alpha"]]), np.array([d["beta"]]), S0=S_old)
    assert np.array_equal(S, np.array(d["S_new"]))
    assert np.array_equal(o[0], np.array(d["readback_along_k"]))
    o2, S2 = rc.unified(q, k, v, np.log(np.array([d["alpha"]])), beta=np.array([d["beta"]]),
                        S0=S_old)
    assert np.array_equal(S2, np.array(d["S_new"]))
    assert np.array_equal(o2[0], np.array(d["readback_along_k"]))
    o3, S3 = native.recurrence(q[None, :, None], k[None, :, None], v[None, :, None],
                               np.zeros((1, 1, 1)), beta=np.ones((1, 1, 1)),
                               h0=S_old[None, None])
    assert np.array_equal(S3[0, 0], np.array(d["S_new"]))
    assert np.array_equal(o3[0, 0, 0], np.array(d["readback_along_k"]))


def test_key_scaling_write_x10_correction_x100():
    d = json.load(open(os.path.join(GOLDEN, "worked_example.json")))["key_scaling"]
    rng = np.random.default_rng(11)
    dk, dv = 4, 3
    S_old = rng.standard_normal((dk, dv))
    k = rng.standard_normal(dk)
    v = rng.standard_normal(dv)

    def delta(kk, vv):
        _, S = rc.gdn_llms_ch11(kk[None], kk[None], vv[None], np.ones(1), np.array([0.7]),
                                S0=S_old)
        return S - S_old

    f = d["factor"]
    corr1, corr10 = delta(k, 0 * v), delta(f * k, 0 * v)
    write1, write10 = delta(k, v) - corr1, delta(f * k, v) - corr10
    np.testing.assert_allclose(write10, d["write_gain"] * write1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(corr10, d["correction_gain"] * corr1, rtol=1e-12, atol=1e-12)
    # and therefore the whole increment is not a uniform rescaling
    full1, full10 = delta(k, v), delta(f * k, v)
    ratio = full10 / full1
    assert np.ptp(ratio) > 1.0


# --------------------------------------------------------------------------
# ch. 11 sections 11.4 and 11.6: recurrence vs closed-form product expansion
# --------------------------------------------------------------------------
@pytest.mark.parametrize("flags", [0, rc.DECAY_CHANNEL, rc.QMIX,
                                   rc.DECAY_CHANNEL | rc.ERASE_CHANNEL | rc.WRITE_CHANNEL])
@pytest.mark.parametrize("with_s0", [False, True])
def test_product_expansion_six_tokens_width_three(flags, with_s0):
    rng = np.random.default_rng(1949)   # the seed the chapter reports
    T, d = 6, 3
    s = seq(rng, T, d, d, channel=bool(flags & rc.DECAY_CHANNEL), s0=with_s0)
    As, Us = ex.transition_matrices(s["q"], s["k"], s["v"], s["g"], s["beta"], s["lam"],
                                    s["b"], s["w"], flags)
    states = ex.expanded_states(As, Us, s["S0"])
    for t in range(T):
        _, S = rc.unified(s["q"][:t + 1], s["k"][:t + 1], s["v"][:t + 1], s["g"][:t + 1],
                          s["beta"][:t + 1], s["lam"][:t + 1], s["b"][:t + 1], s["w"][:t + 1],
                          s["S0"], 1.0, flags)
        # the chapter reports a 4.44e-16 maximum error for this check
        assert np.max(np.abs(S - states[t])) <= 4e-15


# --------------------------------------------------------------------------
# ch. 11 section 11.6: unit key with beta = 1 overwrites with error 0
# --------------------------------------------------------------------------
def test_unit_key_overwrite_error_zero():
    S_old = np.array([[2.0, -1.0, 4.0], [7.0, 0.0, -3.0], [1.0, 5.0, 6.0]])
    k = np.array([[0.0, 1.0, 0.0]])
    v = np.array([[9.0, -8.0, 2.0]])
    for S in (rc.gdn_llms_ch11(k, k, v, np.ones(1), np.ones(1), S0=S_old)[1],
              rc.unified(k, k, v, np.zeros(1), beta=np.ones(1), S0=S_old)[1],
              native.recurrence(k[None, :, None], k[None, :, None], v[None, :, None],
                                np.zeros((1, 1, 1)), beta=np.ones((1, 1, 1)),
                                h0=S_old[None, None])[1][0, 0]):
        assert np.array_equal(S[1], v[0])
        assert np.array_equal(S[[0, 2]], S_old[[0, 2]])


# --------------------------------------------------------------------------
# Reductions between the pages' variants (Gated DeltaNet-2 notes, key
# design 1; Q-Delta notes, key design 3 and the GatedDeltaNet comparison)
# --------------------------------------------------------------------------
def test_gdn2_with_b_w_equal_beta_is_kda():
    rng = np.random.default_rng(1)
    T, dk, dv = 20, 5, 3
    s = seq(rng, T, dk, dv, channel=True)
    alpha = np.exp(s["g"])
    bb = np.repeat(s["beta"][:, None], dk, 1)
    ww = np.repeat(s["beta"][:, None], dv, 1)
    o2, S2 = rc.gdn2_decoupled(s["q"], s["k"], s["v"], alpha, bb, ww, s["S0"], scale=0.4)
    ok, Sk = rc.kda_kimi(s["q"], s["k"], s["v"], alpha, s["beta"], s["S0"].T, scale=0.4)
    assert relerr(o2, ok) <= 1e-13
    assert relerr(S2, Sk.T) <= 1e-13


def test_kda_with_uniform_channels_is_gated_deltanet():
    rng = np.random.default_rng(2)
    T, dk, dv = 20, 5, 3
    s = seq(rng, T, dk, dv)
    alpha = np.exp(s["g"])
    ok, Sk = rc.kda_kimi(s["q"], s["k"], s["v"], np.repeat(alpha[:, None], dk, 1), s["beta"],
                         s["S0"].T)
    og, Sg = rc.gdn_llms_ch11(s["q"], s["k"], s["v"], alpha, s["beta"], s["S0"])
    assert relerr(ok, og) <= 1e-13
    assert relerr(Sk.T, Sg) <= 1e-13


def test_qdelta_with_lambda_zero_is_gated_deltanet():
    rng = np.random.default_rng(3)
    T, dk, dv = 20, 5, 3
    s = seq(rng, T, dk, dv)
    alpha = np.exp(s["g"])
    oq, Sq = rc.qdelta_q_delta_page(s["q"], s["k"], s["v"], alpha, s["beta"], np.zeros(T),
                                    s["S0"].T)
    og, Sg = rc.gdn_llms_ch11(s["q"], s["k"], s["v"], alpha, s["beta"], s["S0"])
    assert relerr(oq, og) <= 1e-13
    assert relerr(Sq.T, Sg) <= 1e-13
    # and lambda != 0 really changes the result
    oq2, _ = rc.qdelta_q_delta_page(s["q"], s["k"], s["v"], alpha, s["beta"], s["lam"],
                                    s["S0"].T)
    assert relerr(oq2, og) > 1e-3


def _page_oracle(flags, s, scale):
    """The per-page formulation matching a flag set, in d_k x d_v terms."""
    alpha = np.exp(s["g"])
    dk, dv = s["k"].shape[1], s["v"].shape[1]
    if flags == 0:
        return rc.gdn_llms_ch11(s["q"], s["k"], s["v"], alpha, s["beta"], s["S0"], scale)
    if flags == rc.DECAY_CHANNEL:
        o, S = rc.kda_kimi(s["q"], s["k"], s["v"], alpha, s["beta"], s["S0"].T, scale)
        return o, S.T
    if flags == rc.QMIX:
        o, S = rc.qdelta_q_delta_page(s["q"], s["k"], s["v"], alpha, s["beta"], s["lam"],
                                      s["S0"].T, scale)
        return o, S.T
    # Gated DeltaNet-2 and its partial ablations (scalar b or scalar w = beta)
    a = alpha if flags & rc.DECAY_CHANNEL else np.repeat(alpha[:, None], dk, 1)
    bb = s["b"] if flags & rc.ERASE_CHANNEL else np.repeat(s["beta"][:, None], dk, 1)
    ww = s["w"] if flags & rc.WRITE_CHANNEL else np.repeat(s["beta"][:, None], dv, 1)
    return rc.gdn2_decoupled(s["q"], s["k"], s["v"], a, bb, ww, s["S0"], scale)


@pytest.mark.parametrize("flags", [0, rc.DECAY_CHANNEL, rc.QMIX,
                                   rc.DECAY_CHANNEL | rc.ERASE_CHANNEL | rc.WRITE_CHANNEL,
                                   rc.ERASE_CHANNEL, rc.WRITE_CHANNEL,
                                   rc.DECAY_CHANNEL | rc.ERASE_CHANNEL])
def test_unified_form_matches_each_page(flags):
    rng = np.random.default_rng(100 + flags)
    s = seq(rng, 25, 6, 4, channel=bool(flags & rc.DECAY_CHANNEL))
    o_p, S_p = _page_oracle(flags, s, 0.37)
    o_u, S_u = rc.unified(s["q"], s["k"], s["v"], s["g"], s["beta"], s["lam"], s["b"], s["w"],
                          s["S0"], 0.37, flags)
    assert relerr(o_u, o_p) <= 1e-13
    assert relerr(S_u, S_p) <= 1e-13


# --------------------------------------------------------------------------
# Q-Delta notes, key design 4: Lemma 3.1 (one-step contraction)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("decay", [False, True])
def test_qdelta_lemma_3_1(decay):
    rng = np.random.default_rng(31)
    T, dk, dv = 30, 6, 4
    s = seq(rng, T, dk, dv)
    alpha = np.exp(s["g"]) if decay else np.ones(T)
    x_all = s["k"] + s["lam"][:, None] * s["q"]
    a_all = np.sum(s["k"] * x_all, 1)
    beta = s["beta"] * np.minimum(1.0, 1.9 / a_all)          # keeps beta*a in (0, 2)
    S = s["S0"].T.copy()                                       # page orientation d_v x d_k
    for t in range(T):
        _, S_new = rc.qdelta_q_delta_page(s["q"][t:t + 1], s["k"][t:t + 1], s["v"][t:t + 1],
                                          alpha[t:t + 1], beta[t:t + 1], s["lam"][t:t + 1], S)
        x, a = x_all[t], a_all[t]
        assert 0.0 < beta[t] * a < 2.0
        after = np.linalg.norm(s["v"][t] - S_new @ x)
        before = np.linalg.norm(s["v"][t] - alpha[t] * S @ x)   # S~ = alpha S_{t-1}
        assert abs(after - abs(1 - beta[t] * a) * before) <= 1e-13 * max(1.0, before)
        assert after <= before + 1e-13
        S = S_new


# --------------------------------------------------------------------------
# KDA derivation, section 2.1: read-back of the written key, locality
# --------------------------------------------------------------------------
def test_readback_and_orthogonal_locality():
    rng = np.random.default_rng(21)
    dk, dv = 6, 4
    S0 = rng.standard_normal((dk, dv))
    k = _unit(rng.standard_normal(dk))
    v = rng.standard_normal(dv)
    beta = 0.35
    x = rng.standard_normal(dk)
    x -= (x @ k) * k                                          # x orthogonal to k
    _, S1 = rc.unified(k[None], k[None], v[None], np.zeros(1), beta=np.array([beta]), S0=S0)
    np.testing.assert_allclose(S1.T @ k, (1 - beta) * (S0.T @ k) + beta * v, rtol=0, atol=1e-14)
    np.testing.assert_allclose(S1.T @ x, S0.T @ x, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# ch. 11 section 11.6 exercises: alpha = 0, beta = 0
# --------------------------------------------------------------------------
def test_alpha_zero_keeps_only_current_write():
    rng = np.random.default_rng(5)
    s = seq(rng, 1, 5, 3)
    _, S = rc.unified(s["q"], s["k"], s["v"], np.array([-np.inf]), s["beta"], S0=s["S0"])
    np.testing.assert_allclose(S, s["beta"][0] * np.outer(s["k"][0], s["v"][0]), rtol=1e-15)


def test_beta_zero_still_reads_decayed_state():
    rng = np.random.default_rng(6)
    s = seq(rng, 1, 5, 3)
    o, S = rc.unified(s["q"], s["k"], s["v"], s["g"], np.zeros(1), S0=s["S0"], scale=0.5)
    a = np.exp(s["g"][0])
    np.testing.assert_allclose(S, a * s["S0"], rtol=1e-15)
    np.testing.assert_allclose(o[0], a * s["S0"].T @ (0.5 * s["q"][0]), rtol=1e-14)
    assert np.max(np.abs(o)) > 1e-3


# --------------------------------------------------------------------------
# KDA derivation, section 1.1: with no erase the rule is (decayed) linear
# attention, a masked matmul computed here without any recurrence
# --------------------------------------------------------------------------
@pytest.mark.parametrize("decay", ["none", "scalar", "channel"])
def test_no_erase_is_masked_linear_attention(decay):
    rng = np.random.default_rng(7)
    T, dk, dv = 40, 6, 4
    s = seq(rng, T, dk, dv, channel=(decay == "channel"))
    g = {"none": np.zeros((T, dk)), "scalar": np.repeat(s["g"][:, None], dk, 1),
         "channel": s["g"]}[decay]
    scale = 0.6
    flags = rc.DECAY_CHANNEL | rc.ERASE_CHANNEL | rc.WRITE_CHANNEL
    o, S = rc.unified(s["q"], s["k"], s["v"], g, b=np.zeros((T, dk)), w=np.ones((T, dv)),
                      S0=s["S0"], scale=scale, flags=flags)
    G = np.cumsum(g, axis=0)                                   # [T, dk]
    # weights[t, i] = sum_c scale q_tc k_ic exp(G_tc - G_ic) for i <= t
    weights = np.einsum("tc,ic,tic->ti", scale * s["q"], s["k"],
                        np.exp(G[:, None, :] - G[None, :, :]))
    o_ref = np.tril(weights) @ s["v"] + (scale * s["q"] * np.exp(G)) @ s["S0"]
    assert relerr(o, o_ref) <= 1e-12
    if decay == "none":
        o_plain = np.tril(scale * s["q"] @ s["k"].T) @ s["v"] + scale * s["q"] @ s["S0"]
        assert relerr(o, o_plain) <= 1e-12


# --------------------------------------------------------------------------
# Gated DeltaNet-2 notes, key design 1: the update is the stationary point of
# L_t(S) = ||S - S_bar||_F^2 - 2 <S^T k, z - S_bar^T e>  (finite differences)
# --------------------------------------------------------------------------
def test_fast_weight_objective_is_stationary_at_update():
    rng = np.random.default_rng(8)
    dk, dv = 5, 3
    s = seq(rng, 1, dk, dv, channel=True)
    alpha = np.exp(s["g"][0])
    _, S_t = rc.gdn2_decoupled(s["q"], s["k"], s["v"], alpha[None], s["b"], s["w"], s["S0"])
    S_bar = np.diag(alpha) @ s["S0"]
    e = s["b"][0] * s["k"][0]
    z = s["w"][0] * s["v"][0]

    def L(S):
        return np.sum((S - S_bar) ** 2) - 2.0 * np.dot(S.T @ s["k"][0], z - S_bar.T @ e)

    h = 1e-5
    grad = np.zeros_like(S_t)
    for i in range(dk):
        for j in range(dv):
            E = np.zeros_like(S_t)
            E[i, j] = h
            grad[i, j] = (L(S_t + E) - L(S_t - E)) / (2 * h)
    assert np.max(np.abs(grad)) <= 1e-8
    # a perturbed state is not stationary (the check has teeth)
    assert np.max(np.abs(2 * (S_t + 0.01 - S_bar) - 2 * np.outer(s["k"][0], z - S_bar.T @ e))) > 1e-3


# KDA derivation, section 2.2: DeltaNet is one gradient step of size beta on
# 1/2 ||S^T k - v||^2 (d_k x d_v orientation), again with a numeric gradient
def test_delta_rule_is_one_gradient_step():
    rng = np.random.default_rng(9)
    dk, dv = 5, 3
    s = seq(rng, 1, dk, dv)
    k, v, beta, S0 = s["k"][0], s["v"][0], s["beta"][0], s["S0"]

    def L(S):
        r = S.T @ k - v
        return 0.5 * r @ r

    h = 1e-5
    grad = np.zeros_like(S0)
    for i in range(dk):
        for j in range(dv):
            E = np.zeros_like(S0)
            E[i, j] = h
            grad[i, j] = (L(S0 + E) - L(S0 - E)) / (2 * h)
    _, S1 = rc.gdn_llms_ch11(s["q"], s["k"], s["v"], np.ones(1), s["beta"], S0)
    np.testing.assert_allclose(S1, S0 - beta * grad, rtol=0, atol=1e-9)


# --------------------------------------------------------------------------
# Gated DeltaNet-2 notes, key design 2: the chunk algebra reaches the token
# recurrence, for any chunk size, ragged tails and every flag combination
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
@pytest.mark.parametrize("C", [1, 16, 64])
def test_chunked_equals_token_recurrence(T, C):
    for flags in (0, rc.DECAY_CHANNEL, rc.QMIX, rc.DECAY_CHANNEL | rc.ERASE_CHANNEL | rc.WRITE_CHANNEL):
        rng = np.random.default_rng(1000 * T + C + flags)
        s = seq(rng, T, 8, 6, channel=bool(flags & rc.DECAY_CHANNEL))
        args = (s["q"], s["k"], s["v"], s["g"], s["beta"], s["lam"], s["b"], s["w"], s["S0"],
                0.35, flags)
        o_t, S_t = rc.unified(*args)
        o_c, S_c = ch.chunked(*args, C=C)
        assert relerr(o_c, o_t) <= 1e-12, flags
        assert relerr(S_c, S_t) <= 1e-12, flags


def test_chunked_with_workload_decay_ranges():
    # channel decay -exp(N(-2, 0.5)) and scalar -softplus(N(0,1)) at C = 64
    rng = np.random.default_rng(77)
    T, dk, dv = 130, 16, 8
    s = seq(rng, T, dk, dv, channel=True)
    s["g"] = -np.exp(rng.normal(-2.0, 0.5, size=(T, dk)))
    flags = rc.DECAY_CHANNEL | rc.ERASE_CHANNEL | rc.WRITE_CHANNEL
    args = (s["q"], s["k"], s["v"], s["g"], s["beta"], s["lam"], s["b"], s["w"], s["S0"],
            dk ** -0.5, flags)
    assert relerr(ch.chunked(*args)[0], rc.unified(*args)[0]) <= 1e-12


def test_forward_substitution_inverts_unit_lower_triangular():
    rng = np.random.default_rng(12)
    T = np.tril(rng.standard_normal((64, 64)) * 0.2, -1)
    A = ch.forward_substitution_inverse(T)
    np.testing.assert_allclose(A @ (np.eye(64) + T), np.eye(64), atol=1e-12)
    np.testing.assert_allclose(A, np.linalg.inv(np.eye(64) + T), atol=1e-12)


def test_chunk_local_cumsum_is_a_cumsum_per_chunk():
    rng = np.random.default_rng(13)
    g = rng.standard_normal((130, 4))
    G = ch.chunk_local_cumsum(g, 64)
    for n0 in (0, 64, 128):
        np.testing.assert_allclose(G[n0:n0 + 64], np.cumsum(g[n0:n0 + 64], axis=0), rtol=1e-15)


# --------------------------------------------------------------------------
# ch. 11 section 11.3: streaming. Returning the final state and passing it
# back as the initial state continues the sequence.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("split", [1, 40, 64, 99])
def test_streaming_split_equals_whole(split):
    rng = np.random.default_rng(14)
    s = seq(rng, 130, 8, 6, channel=True)
    flags = rc.DECAY_CHANNEL | rc.QMIX
    cut = lambda a, sl: a[sl]
    full = rc.unified(s["q"], s["k"], s["v"], s["g"], s["beta"], s["lam"], None, None, s["S0"],
                      0.5, flags)
    p1 = slice(0, split)
    p2 = slice(split, None)
    o1, S1 = rc.unified(*(cut(s[x], p1) for x in ("q", "k", "v", "g", "beta", "lam")),
                        None, None, s["S0"], 0.5, flags)
    o2, S2 = rc.unified(*(cut(s[x], p2) for x in ("q", "k", "v", "g", "beta", "lam")),
                        None, None, S1, 0.5, flags)
    assert np.array_equal(np.concatenate([o1, o2]), full[0])
    assert np.array_equal(S2, full[1])
    # the chunked oracle restarted mid-chunk agrees too
    o1c, S1c = ch.chunked(*(cut(s[x], p1) for x in ("q", "k", "v", "g", "beta", "lam")),
                          None, None, s["S0"], 0.5, flags)
    o2c, S2c = ch.chunked(*(cut(s[x], p2) for x in ("q", "k", "v", "g", "beta", "lam")),
                          None, None, S1c, 0.5, flags)
    assert relerr(np.concatenate([o1c, o2c]), full[0]) <= 1e-12
    assert relerr(S2c, full[1]) <= 1e-12


# --------------------------------------------------------------------------
# The C oracle against the pinned numpy oracle, every flag combination
# --------------------------------------------------------------------------
@pytest.mark.parametrize("flags", ALL_FLAGS)
def test_native_oracle_matches_numpy(flags):
    rng = np.random.default_rng(500 + flags)
    B, T, H, dk, dv = 2, 37, 3, 8, 5
    chan = bool(flags & rc.DECAY_CHANNEL)
    q = _unit(rng.standard_normal((B, T, H, dk)))
    k = _unit(rng.standard_normal((B, T, H, dk)))
    v = rng.standard_normal((B, T, H, dv))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, H, dk) if chan else (B, T, H))))
    beta = _sig(rng.standard_normal((B, T, H)))
    lam = rng.uniform(size=(B, T, H))
    b = _sig(rng.standard_normal((B, T, H, dk)))
    w = _sig(rng.standard_normal((B, T, H, dv)))
    h0 = 0.2 * rng.standard_normal((B, H, dk, dv))
    o_n, h_n = native.recurrence(q, k, v, g, beta, lam, b, w, h0, 0.45, flags, nthreads=2)
    o_p, h_p = rc.unified_batched(q, k, v, g, beta, lam, b, w, h0, 0.45, flags)
    assert relerr(o_n, o_p) <= 1e-13
    assert relerr(h_n, h_p) <= 1e-13


def test_native_oracle_rejects_missing_gates():
    z = np.zeros((1, 2, 1, 4))
    with pytest.raises(ValueError):
        native.recurrence(z, z, z, np.zeros((1, 2, 1)), beta=None, flags=0)
    with pytest.raises(ValueError):
        native.recurrence(z, z, z, np.zeros((1, 2, 1)), beta=np.zeros((1, 2, 1)),
                          flags=rc.QMIX)


# --------------------------------------------------------------------------
# The pins have teeth: mistakes planted in the oracle (on the CPU) fail them
# --------------------------------------------------------------------------
def test_planted_mistakes_are_caught(monkeypatch):
    rng = np.random.default_rng(15)
    s = seq(rng, 20, 6, 4, channel=True)
    real = rc.erase_write_vectors

    def run(flags):
        o_p, _ = _page_oracle(flags, s, 0.5)
        o_u, _ = rc.unified(s["q"], s["k"], s["v"], s["g"], s["beta"], s["lam"], s["b"],
                            s["w"], s["S0"], 0.5, flags)
        return relerr(o_u, o_p)

    def lam_sign(q, k, v, beta, lam, b, w, flags):          # x = k - lam q
        return real(q, k, v, beta, -lam, b, w, flags)

    def drop_write_gate(q, k, v, beta, lam, b, w, flags):   # z = beta v under WRITE_CHANNEL
        return real(q, k, v, beta, lam, b, w, flags & ~rc.WRITE_CHANNEL)

    monkeypatch.setattr(rc, "erase_write_vectors", lam_sign)
    assert run(rc.QMIX) > 1e-3
    monkeypatch.setattr(rc, "erase_write_vectors", drop_write_gate)
    assert run(rc.DECAY_CHANNEL | rc.ERASE_CHANNEL | rc.WRITE_CHANNEL) > 1e-3
    monkeypatch.setattr(rc, "erase_write_vectors", real)
    assert run(rc.QMIX) <= 1e-13

    # a first-order stand-in for (I + T)^{-1} breaks the chunk algebra
    monkeypatch.setattr(ch, "forward_substitution_inverse",
                        lambda T: np.eye(T.shape[0]) - T)
    args = (s["q"], s["k"], s["v"], s["g"], s["beta"], s["lam"], s["b"], s["w"], s["S0"],
            0.5, rc.DECAY_CHANNEL)
    assert relerr(ch.chunked(*args, C=16)[0], rc.unified(*args)[0]) > 1e-3

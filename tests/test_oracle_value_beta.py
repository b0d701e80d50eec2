"""Pins of the per-value-channel write strength (the README variant of the
LLMs-from-scratch Gated DeltaNet chapter, section 11.3).

The chapter says the README module scales the prediction error channel by
channel with a write gate per value channel, keeps one scalar forget gate per
head, and (section 11.4) that each state column then follows its own affine
update. The pins: a hand-worked overwrite, the column decomposition into
scalar-gate Gated DeltaNet runs, the reduction to Gated DeltaNet when the gate
is equal across channels, the unified form and the C oracle against the page's
own form, and planted mistakes that fail them.
"""
import numpy as np
import pytest

from oracle import native
from oracle import recurrence as rc

BC = rc.BETA_CHANNEL


def _seq(seed, T=23, dk=6, dv=5):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    alpha = np.exp(-np.log1p(np.exp(rng.standard_normal(T))))
    beta_v = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, dv))))
    S0 = 0.3 * rng.standard_normal((dk, dv))
    return q, k, v, alpha, beta_v, S0


def test_hand_worked_overwrite_per_channel():
    # k = e_1, alpha = 1: row 1 of S moves by beta_v toward v, row 2 is kept
    a, b, c, d = 0.7, -1.1, 0.4, 2.0
    S0 = np.array([[a, b], [c, d]])
    k = np.array([[1.0, 0.0]])
    v = np.array([[3.0, 4.0]])
    q = np.array([[0.0, 1.0]])
    o, S = rc.gdn_value_beta_ch11(q, k, v, np.ones(1), np.array([[1.0, 0.5]]), S0)
    np.testing.assert_allclose(S, [[3.0, (b + 4.0) / 2.0], [c, d]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(o[0], [c, d], rtol=0, atol=1e-15)   # reads row 2


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_each_state_column_is_a_scalar_gate_gated_deltanet(seed):
    q, k, v, alpha, beta_v, S0 = _seq(seed)
    o, S = rc.gdn_value_beta_ch11(q, k, v, alpha, beta_v, S0, scale=0.4)
    for j in range(v.shape[1]):
        oj, Sj = rc.gdn_llms_ch11(q, k, v[:, j:j + 1], alpha, beta_v[:, j], S0[:, j:j + 1],
                                  scale=0.4)
        np.testing.assert_allclose(o[:, j], oj[:, 0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(S[:, j], Sj[:, 0], rtol=1e-12, atol=1e-13)


def test_equal_gate_across_channels_is_gated_deltanet():
    q, k, v, alpha, beta_v, S0 = _seq(3)
    beta = beta_v[:, 0]
    o, S = rc.gdn_value_beta_ch11(q, k, v, alpha, np.repeat(beta[:, None], v.shape[1], 1), S0)
    o2, S2 = rc.gdn_llms_ch11(q, k, v, alpha, beta, S0)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, S2, rtol=1e-12, atol=1e-13)


def test_unified_form_and_c_oracle_match_the_page():
    q, k, v, alpha, beta_v, S0 = _seq(4)
    o, S = rc.gdn_value_beta_ch11(q, k, v, alpha, beta_v, S0, scale=0.5)
    g = np.log(alpha)
    o2, S2 = rc.unified(q, k, v, g, beta=beta_v, S0=S0, scale=0.5, flags=BC)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, S2, rtol=1e-12, atol=1e-13)
    o3, S3 = native.recurrence(q[None, :, None], k[None, :, None], v[None, :, None],
                               g[None, :, None], beta=beta_v[None, :, None], h0=S0[None, None],
                               scale=0.5, flags=BC)
    np.testing.assert_allclose(o3[0, :, 0], o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S3[0, 0], S, rtol=1e-12, atol=1e-13)


def test_c_oracle_with_channel_decay_matches_numpy():
    rng = np.random.default_rng(5)
    B, T, H, dk, dv = 2, 19, 2, 8, 4
    q, k = rng.standard_normal((2, B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    g = -np.exp(rng.standard_normal((B, T, H, dk)) - 2)
    beta = rng.random((B, T, H, dv))
    h0 = rng.standard_normal((B, H, dk, dv))
    flags = BC | rc.DECAY_CHANNEL
    o, hT = native.recurrence(q, k, v, g, beta=beta, h0=h0, scale=0.7, flags=flags)
    o2, hT2 = rc.unified_batched(q, k, v, g, beta=beta, h0=h0, scale=0.7, flags=flags)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hT, hT2, rtol=1e-12, atol=1e-12)


def test_planted_mistakes_fail_the_pins(monkeypatch):
    q, k, v, alpha, beta_v, S0 = _seq(6)
    g = np.log(alpha)
    want = rc.gdn_value_beta_ch11(q, k, v, alpha, beta_v, S0)[0]
    real = rc.erase_write_vectors

    # the gate on the write only (z = beta (.) v, erase unscaled): a GDN-2-like write gate
    def write_only(q_, k_, v_, beta, lam, b, w, flags):
        return (k_, beta * v_) if flags & BC else real(q_, k_, v_, beta, lam, b, w, flags)

    monkeypatch.setattr(rc, "erase_write_vectors", write_only)
    monkeypatch.setattr(rc, "BETA_CHANNEL", 0)       # and no per-channel error scaling
    got = rc.unified(q, k, v, g, beta=beta_v, S0=S0, flags=BC)[0]
    assert np.abs(got - want).max() > 1e-3

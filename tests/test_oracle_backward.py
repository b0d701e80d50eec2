"""Pins of the gradient oracle (oracle/backward.py).

* Autograd against central finite differences of the forward recurrence
  (directional derivatives along random directions), every flag combination
  and the per-value-channel write strength: pins the autograd form to the
  forward oracle by a route that shares no differentiation code with it.
* The chunkwise backward of the Gated DeltaNet-2 notes (key design 3) against
  autograd, every flag combination, chunk sizes 1, 4 and 16, ragged lengths.
* Special case: beta = 0 writes nothing, so the values get no gradient.
* Planted mistakes in the notes' two formulas (the gates pulled out of dA as a
  scalar, the diagonal kept in dT) fail against autograd.
"""
import numpy as np
import pytest

from oracle import backward as bw
from oracle import recurrence as rc

FLAGS = list(range(16)) + [rc.BETA_CHANNEL]


def _inputs(flags, T=9, dk=4, dv=3, seed=0):
    rng = np.random.default_rng(seed + 101 * flags)
    k = rng.standard_normal((T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    x = dict(q=rng.standard_normal((T, dk)) * 0.7, k=k, v=rng.standard_normal((T, dv)),
             g=(-rng.random((T, dk)) * 0.6 if flags & rc.DECAY_CHANNEL else -rng.random(T) * 0.6),
             S0=rng.standard_normal((dk, dv)) * 0.3, scale=0.8, flags=flags)
    if flags & rc.BETA_CHANNEL:
        x["beta"] = rng.random((T, dv))
    elif not (flags & rc.ERASE_CHANNEL and flags & rc.WRITE_CHANNEL):
        x["beta"] = rng.random(T)
    if flags & rc.QMIX:
        x["lam"] = rng.random(T)
    if flags & rc.ERASE_CHANNEL:
        x["b"] = rng.random((T, dk))
    if flags & rc.WRITE_CHANNEL:
        x["w"] = rng.random((T, dv))
    cot = dict(dO=rng.standard_normal((T, dv)), dST=rng.standard_normal((dk, dv)))
    return x, cot


def _loss(x, cot):
    o, S = rc.unified(x["q"], x["k"], x["v"], x["g"], x.get("beta"), x.get("lam"), x.get("b"),
                      x.get("w"), x["S0"], x["scale"], x["flags"])
    return float((cot["dO"] * o).sum() + (cot["dST"] * S).sum())


@pytest.mark.parametrize("flags", FLAGS)
def test_autograd_matches_finite_differences(flags):
    x, cot = _inputs(flags)
    grads = bw.grad_autograd(**x, **cot)
    rng = np.random.default_rng(7)
    names = [n for n in bw.NAMES if x.get(n) is not None]
    for _ in range(3):
        u = {n: rng.standard_normal(np.shape(x[n])) for n in names}
        eps = 1e-6
        xp = dict(x, **{n: x[n] + eps * u[n] for n in names})
        xm = dict(x, **{n: x[n] - eps * u[n] for n in names})
        fd = (_loss(xp, cot) - _loss(xm, cot)) / (2 * eps)
        an = sum(float((grads[n] * u[n]).sum()) for n in names)
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (fd, an)


@pytest.mark.parametrize("C", [1, 4, 16])
@pytest.mark.parametrize("T", [13, 16, 17])
@pytest.mark.parametrize("flags", range(16))
def test_chunked_backward_matches_autograd(flags, T, C):
    x, cot = _inputs(flags, T=T, dk=5, dv=4, seed=T + C)
    a = bw.grad_autograd(**x, **cot)
    c = bw.chunked_backward(**x, **cot, C=C)
    for n in bw.NAMES:
        if a[n] is None:
            assert c[n] is None, n
            continue
        np.testing.assert_allclose(c[n], a[n], rtol=1e-9, atol=1e-11, err_msg=n)


def test_zero_write_strength_gives_values_no_gradient():
    x, cot = _inputs(0)
    x["beta"] = np.zeros_like(x["beta"])
    for grads in (bw.grad_autograd(**x, **cot), bw.chunked_backward(**x, **cot, C=4)):
        assert np.abs(grads["v"]).max() == 0.0


def _max_rel(a, c):
    return max(np.abs(a[n] - c[n]).max() / max(np.abs(a[n]).max(), 1e-30)
               for n in bw.NAMES if a[n] is not None)


def test_planted_mistakes_fail(monkeypatch):
    x, cot = _inputs(rc.DECAY_CHANNEL | rc.ERASE_CHANNEL | rc.WRITE_CHANNEL, T=17, dk=5, dv=4)
    a = bw.grad_autograd(**x, **cot)
    assert _max_rel(a, bw.chunked_backward(**x, **cot, C=8)) < 1e-9
    real_dA, real_dT = bw.gate_aware_dA, bw.inverse_adjoint

    # scalar post-scaling, which the notes rule out for per-channel gates: each
    # row's gates treated as one scalar (the channel mean) when forming dA
    def scalar_dA(dU, Z, dY, E_bar):
        rowwise = lambda M: np.repeat(M.mean(axis=1, keepdims=True), M.shape[1], axis=1)
        return dU @ rowwise(Z).T + dY @ rowwise(E_bar).T

    monkeypatch.setattr(bw, "gate_aware_dA", scalar_dA)
    assert _max_rel(a, bw.chunked_backward(**x, **cot, C=8)) > 1e-3
    monkeypatch.setattr(bw, "gate_aware_dA", real_dA)

    # the diagonal kept in the adjoint of the inverse
    monkeypatch.setattr(bw, "inverse_adjoint", lambda A, dA: -np.tril(A.T @ dA @ A.T, 0))
    assert _max_rel(a, bw.chunked_backward(**x, **cot, C=8)) > 1e-3
    monkeypatch.setattr(bw, "inverse_adjoint", real_dT)
    assert _max_rel(a, bw.chunked_backward(**x, **cot, C=8)) < 1e-9

"""Pins of the fp64 projector fit step (CPU).

The gradient is checked against central finite differences of the loss, an
Euler identity of the reconstruction (R is homogeneous of degree 2 in P and
in Q), and closed forms for diagonal projectors; the step is checked to
descend.  None of these reuses the gradient formula.
"""

import numpy as np
import pytest

from oracle.lsp import Projector
from oracle.lsp_fit import fit_loss, fit_step, stepped


def _proj(rows, d, k, rng, dup=False):
    idx = np.stack([rng.choice(d, size=k, replace=False) for _ in range(rows)])
    if dup and k > 1:
        idx[::2, 1] = idx[::2, 0]          # a repeated id in every other row
    val = rng.normal(0.0, 1.0 / np.sqrt(k), size=(rows, k))
    return Projector(idx, val, d)


@pytest.mark.parametrize("m,n,d,k,dup,seed", [(7, 5, 3, 2, False, 0), (6, 6, 4, 1, False, 1),
                                               (9, 4, 4, 3, False, 2), (8, 10, 5, 2, True, 3)])
def test_gradient_matches_central_differences(m, n, d, k, dup, seed):
    rng = np.random.default_rng(seed)
    G = rng.normal(size=(m, n))
    P, Q = _proj(m, d, k, rng, dup), _proj(n, d, k, rng, dup)
    res = fit_step(G, P, Q, 0.0)
    h = 1e-6
    for which, A, g in (("P", P, res["gP"]), ("Q", Q, res["gQ"])):
        for r in range(A.rows):
            for t in range(A.k):
                vp, vm = A.val.copy(), A.val.copy()
                vp[r, t] += h
                vm[r, t] -= h
                Ap, Am = Projector(A.idx, vp, d), Projector(A.idx, vm, d)
                if which == "P":
                    fd = (fit_loss(G, Ap, Q) - fit_loss(G, Am, Q)) / (2 * h)
                else:
                    fd = (fit_loss(G, P, Ap) - fit_loss(G, P, Am)) / (2 * h)
                assert abs(fd - g[r, t]) <= 1e-5 * max(1.0, abs(g[r, t])), (which, r, t, fd, g[r, t])


def test_euler_identity_of_the_reconstruction():
    # R(cP, Q) = c^2 R(P, Q), so d/dc L(cP, Q) at c = 1 is -4 <E, R>, and
    # that derivative is sum over stored values of grad * value; same for Q
    rng = np.random.default_rng(5)
    m, n, d, k = 40, 30, 8, 3
    G = rng.normal(size=(m, n))
    P, Q = _proj(m, d, k, rng), _proj(n, d, k, rng)
    res = fit_step(G, P, Q, 0.0)
    Pd, Qd = P.dense(), Q.dense()
    R = Pd @ (Pd.T @ G @ Qd) @ Qd.T
    want = -4.0 * np.sum((G - R) * R)
    assert np.isclose(np.sum(res["gP"] * P.val), want, rtol=1e-10, atol=1e-12)
    assert np.isclose(np.sum(res["gQ"] * Q.val), want, rtol=1e-10, atol=1e-12)


def test_identity_projectors_reconstruct_exactly():
    rng = np.random.default_rng(6)
    d = 6
    G = rng.normal(size=(d, d))
    eye = Projector(np.arange(d)[:, None], np.ones((d, 1)), d)
    res = fit_step(G, eye, eye, 0.1)
    assert res["loss"] == 0.0
    assert np.all(res["gP"] == 0.0) and np.all(res["gQ"] == 0.0)


@pytest.mark.parametrize("c", [0.5, 0.9, 1.3])
def test_scaled_identity_closed_form(c):
    # P = c I, Q = I: R = c^2 G, L = (1 - c^2)^2 ||G||^2, and the gradient of
    # the value on row i is -4 c (1 - c^2) ||G[i, :]||^2
    rng = np.random.default_rng(7)
    d = 5
    G = rng.normal(size=(d, d))
    P = Projector(np.arange(d)[:, None], np.full((d, 1), c), d)
    Q = Projector(np.arange(d)[:, None], np.ones((d, 1)), d)
    res = fit_step(G, P, Q, 0.0)
    assert np.isclose(res["loss"], (1 - c * c) ** 2 * np.sum(G * G), rtol=1e-12)
    want = -4.0 * c * (1 - c * c) * np.sum(G * G, axis=1)
    assert np.allclose(res["gP"][:, 0], want, rtol=1e-12, atol=1e-14)


def test_small_step_descends():
    rng = np.random.default_rng(8)
    m, n, d, k = 64, 48, 16, 2
    G = rng.normal(size=(m, n))
    P, Q = _proj(m, d, k, rng), _proj(n, d, k, rng)
    res = fit_step(G, P, Q, 0.0)
    gnorm2 = np.sum(res["gP"] ** 2) + np.sum(res["gQ"] ** 2)
    lr = 1e-3 * res["loss"] / gnorm2
    P2, Q2 = stepped(P, Q, fit_step(G, P, Q, lr))
    after = fit_loss(G, P2, Q2)
    # first-order prediction: L - lr |g|^2
    assert after < res["loss"]
    assert abs(after - (res["loss"] - lr * gnorm2)) < 0.01 * lr * gnorm2


def test_magnitudes_bound_the_values():
    rng = np.random.default_rng(9)
    G = rng.normal(size=(30, 20))
    P, Q = _proj(30, 6, 2, rng), _proj(20, 6, 2, rng)
    res = fit_step(G, P, Q, 0.0)
    assert np.all(np.abs(res["gP"]) <= res["gP_abs"] * (1 + 1e-12))
    assert np.all(np.abs(res["gQ"]) <= res["gQ_abs"] * (1 + 1e-12))
    assert res["loss"] <= res["loss_abs"]

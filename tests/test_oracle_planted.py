"""The oracle's pins catch plausible mistakes (CPU only).

Each test plants one mistake in a copy of the oracle's arithmetic, on the
CPU, and checks that a pin that holds for the real oracle fails for the
broken one.  Nothing here touches the CUDA path.
"""

import numpy as np
import pytest
import torch

from layer_optimizer_gb300 import synth
from oracle import adamw as oa
from oracle import lsp as ol

HP = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _torch_adamw_theta(th, grads):
    p = torch.nn.Parameter(torch.from_numpy(th.copy()))
    opt = torch.optim.AdamW([p], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"], foreach=False)
    for g in grads:
        p.grad = torch.from_numpy(g.copy())
        opt.step()
    return p.detach().numpy()


def _broken_step(kind):
    def step(state, g, t, lr, beta1, beta2, eps, weight_decay):
        g = np.asarray(g, dtype=np.float64)
        bc1, bc2 = 1 - beta1 ** t, 1 - beta2 ** t
        if kind == "no_bias_correction":
            bc1 = bc2 = 1.0
        if kind == "eps_inside_sqrt":
            m = beta1 * state.m + (1 - beta1) * g
            v = beta2 * state.v + (1 - beta2) * g * g
            state.theta = state.theta * (1 - lr * weight_decay) - lr * (m / bc1) / np.sqrt(v / bc2 + eps)
            state.m, state.v = m, v
            return
        if kind == "coupled_decay":
            g = g + weight_decay * state.theta
            decay = 1.0
        else:
            decay = 1 - lr * weight_decay
        m = beta1 * state.m + (1 - beta1) * g
        v = beta2 * state.v + (1 - beta2) * (g if kind == "v_not_squared" else g * g)
        state.theta = state.theta * decay - lr * (m / bc1) / (np.sqrt(v / bc2) + eps)
        state.m, state.v = m, v
    return step


@pytest.mark.parametrize("kind", ["no_bias_correction", "eps_inside_sqrt", "coupled_decay", "v_not_squared"])
def test_planted_adamw_mistakes_fail_a_pin(kind):
    rng = np.random.default_rng(3)
    th = rng.standard_normal(2000) * 0.02
    grads = [np.abs(rng.standard_normal(2000)) * 1e-3 + 1e-4 for _ in range(3)]
    ref = _torch_adamw_theta(th, grads)
    good, bad = oa.AdamWState(th), oa.AdamWState(th)
    for t, g in enumerate(grads, start=1):
        oa.adamw_step(good, g, t, **HP)
        _broken_step(kind)(bad, g, t, **HP)
    assert np.allclose(good.theta, ref, rtol=1e-12, atol=1e-18)
    assert not np.allclose(bad.theta, ref, rtol=1e-9, atol=1e-15)


def _brute(P, Q, G):
    S = np.zeros((P.d, Q.d))
    for i in range(G.shape[0]):
        for li in range(P.k):
            for j in range(G.shape[1]):
                for lj in range(Q.k):
                    S[P.idx[i, li], Q.idx[j, lj]] += P.val[i, li] * G[i, j] * Q.val[j, lj]
    return S


@pytest.mark.parametrize("kind", ["transposed_G", "Q_for_P", "dropped_value", "wrong_sign"])
def test_planted_compress_mistakes_fail_brute_force(kind):
    rng = np.random.default_rng(4)
    m = n = 12
    d, k = 6, 2
    Pi, Pv = synth.projector(m, d, k, 1)
    Qi, Qv = synth.projector(n, d, k, 2)
    P, Q = ol.Projector(Pi, Pv, d), ol.Projector(Qi, Qv, d)
    G = rng.standard_normal((m, n))
    Pd, Qd = P.dense(), Q.dense()
    broken = {
        "transposed_G": Pd.T @ G.T @ Qd,
        "Q_for_P": Qd.T @ G @ Qd,
        "dropped_value": (Pd != 0).T.astype(float) @ G @ Qd,
        "wrong_sign": -(Pd.T @ G @ Qd),
    }[kind]
    want = _brute(P, Q, G)
    S, _ = ol.compress(P, Q, G)
    assert np.allclose(S, want, rtol=1e-12, atol=1e-12)
    assert not np.allclose(broken, want, rtol=1e-6, atol=1e-9)


def _broken_fit_grads(kind, G, P, Q):
    Pd, Qd = P.dense(), Q.dense()
    S = Pd.T @ G @ Qd
    E = G - Pd @ S @ Qd.T
    if kind == "dropped_term":
        gPd = -2.0 * (E @ Qd @ S.T)
    elif kind == "transposed_S":
        gPd = -2.0 * (E @ Qd @ S + G @ Qd @ Qd.T @ E.T @ Pd)
    else:  # wrong sign of the second term
        gPd = -2.0 * (E @ Qd @ S.T - G @ Qd @ Qd.T @ E.T @ Pd)
    return gPd[np.repeat(np.arange(P.rows), P.k).reshape(P.rows, P.k), P.idx]


@pytest.mark.parametrize("kind", ["dropped_term", "transposed_S", "wrong_sign"])
def test_planted_fit_gradient_mistakes_fail_finite_differences(kind):
    from oracle.lsp_fit import fit_loss, fit_step
    rng = np.random.default_rng(11)
    m, n, d, k = 9, 7, 4, 2
    G = rng.normal(size=(m, n))
    P = ol.Projector(np.stack([rng.choice(d, k, replace=False) for _ in range(m)]), rng.normal(size=(m, k)), d)
    Q = ol.Projector(np.stack([rng.choice(d, k, replace=False) for _ in range(n)]), rng.normal(size=(n, k)), d)
    h = 1e-6
    fd = np.zeros((m, k))
    for r in range(m):
        for t in range(k):
            vp, vm = P.val.copy(), P.val.copy()
            vp[r, t] += h
            vm[r, t] -= h
            fd[r, t] = (fit_loss(G, ol.Projector(P.idx, vp, d), Q) - fit_loss(G, ol.Projector(P.idx, vm, d), Q)) / (2 * h)
    good = fit_step(G, P, Q, 0.0)["gP"]
    bad = _broken_fit_grads(kind, G, P, Q)
    assert np.allclose(good, fd, rtol=1e-5, atol=1e-5)
    assert not np.allclose(bad, fd, rtol=1e-3, atol=1e-3)


@pytest.mark.parametrize("kind", ["divide_by_all_tokens", "no_onehot", "transposed_weight_grad"])
def test_planted_lce_mistakes_fail_the_torch_pin(kind):
    rng = np.random.default_rng(12)
    N, D, V = 10, 6, 9
    H, W = rng.normal(size=(N, D)), rng.normal(size=(V, D)) * 0.3
    y = rng.integers(0, V, size=N)
    y[[1, 4]] = -100
    Z = H @ W.T
    P = np.exp(Z - Z.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    valid = y != -100
    dZ = np.where(valid[:, None], P, 0.0)
    if kind != "no_onehot":
        dZ[np.flatnonzero(valid), y[valid]] -= 1.0
    dZ /= N if kind == "divide_by_all_tokens" else valid.sum()
    dW = (H.T @ dZ)[:, :V].T if kind == "transposed_weight_grad" and D >= V else dZ.T @ H
    if kind == "transposed_weight_grad":
        dW = dW[::-1]                                # rows in the wrong order
    Ht, Wt = torch.tensor(H, requires_grad=True), torch.tensor(W, requires_grad=True)
    torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(y), ignore_index=-100).backward()
    from oracle.lce import lce
    good = lce(H, W, y)
    assert np.allclose(good["dW"], Wt.grad.numpy()) and np.allclose(good["dH"], Ht.grad.numpy())
    assert not (np.allclose(dZ @ W, Ht.grad.numpy()) and np.allclose(dW, Wt.grad.numpy()))

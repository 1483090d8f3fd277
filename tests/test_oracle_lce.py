"""Pins of the fp64 linear cross-entropy (CPU).

Checked against torch's float64 cross-entropy and autograd (a library
routine), central finite differences, the uniform-logit closed form
(L = log V), and the invariants of the softmax gradient.
"""

import numpy as np
import pytest
import torch

from oracle.lce import lce, loss_only


def _case(N, D, V, seed, ignore=0):
    rng = np.random.default_rng(seed)
    H = rng.normal(size=(N, D))
    W = rng.normal(size=(V, D)) * 0.3
    y = rng.integers(0, V, size=N)
    if ignore:
        y[rng.choice(N, size=ignore, replace=False)] = -100
    return H, W, y


@pytest.mark.parametrize("N,D,V,ignore", [(5, 4, 7, 0), (12, 8, 30, 3), (1, 3, 2, 0), (9, 6, 11, 9)])
def test_matches_torch_float64(N, D, V, ignore):
    H, W, y = _case(N, D, V, N + D + V, ignore)
    res = lce(H, W, y)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(y), ignore_index=-100)
    if ignore == N:                                   # every token unlabelled: torch gives nan
        assert res["loss"] == 0.0 and not res["dH"].any() and not res["dW"].any()
        return
    loss.backward()
    assert np.isclose(res["loss"], loss.item(), rtol=1e-12, atol=1e-14)
    assert np.allclose(res["dH"], Ht.grad.numpy(), rtol=1e-10, atol=1e-13)
    assert np.allclose(res["dW"], Wt.grad.numpy(), rtol=1e-10, atol=1e-13)


def test_finite_differences():
    H, W, y = _case(4, 3, 5, 1, ignore=1)
    res = lce(H, W, y)
    h = 1e-6
    for A, g in ((H, res["dH"]), (W, res["dW"])):
        for idx in np.ndindex(A.shape):
            Ap, Am = A.copy(), A.copy()
            Ap[idx] += h
            Am[idx] -= h
            if A is H:
                fd = (loss_only(Ap, W, y) - loss_only(Am, W, y)) / (2 * h)
            else:
                fd = (loss_only(H, Ap, y) - loss_only(H, Am, y)) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-7 * max(1.0, abs(g[idx])), (idx, fd, g[idx])


def test_uniform_logits_closed_form():
    # W = 0: every logit is 0, L = log V, dZ = (1/V - onehot)/N, dH = 0
    N, D, V = 6, 4, 9
    rng = np.random.default_rng(2)
    H = rng.normal(size=(N, D))
    y = rng.integers(0, V, size=N)
    res = lce(H, np.zeros((V, D)), y)
    assert res["loss"] == pytest.approx(np.log(V), rel=1e-15)
    want = np.full((N, V), 1.0 / V)
    want[np.arange(N), y] -= 1.0
    assert np.allclose(res["dZ"], want / N, rtol=1e-14, atol=1e-17)
    assert not res["dH"].any()
    assert np.allclose(res["dW"], (want / N).T @ H, rtol=1e-13, atol=1e-16)


def test_gradient_rows_sum_to_zero_and_ignored_rows_are_zero():
    H, W, y = _case(10, 5, 13, 4, ignore=4)
    res = lce(H, W, y)
    assert np.allclose(res["dZ"].sum(axis=1), 0.0, atol=1e-15)
    assert not res["dZ"][y == -100].any()
    assert res["n"] == 6
    assert np.all(np.abs(res["dH"]) <= res["dH_abs"] * (1 + 1e-12))
    assert np.all(np.abs(res["dW"]) <= res["dW_abs"] * (1 + 1e-12))


@pytest.mark.parametrize("N,D,V,chunk,ignore", [(7, 5, 33, 8, 2), (16, 4, 100, 100, 0), (3, 6, 17, 5, 3)])
def test_chunked_lse_and_sampled_rows_match_the_whole_row_oracle(N, D, V, chunk, ignore):
    # the sampled form the full-size checks use: the per-token log-sum-exp
    # over vocabulary chunks, then dH rows and dW rows from it, against the
    # oracle that holds every logit (ragged last chunk, unlabelled tokens)
    from oracle.lce import lce_rows, token_lse
    H, W, y = _case(N, D, V, 100 + N + V, ignore)
    full = lce(H, W, y)
    lse = token_lse(H, W, chunk=chunk)
    assert np.allclose(lse, full["lse"], rtol=1e-13, atol=1e-13)
    trows = [0, N - 1, N // 2]
    vrows = [0, V - 1, V // 3, int(y[y != -100][0]) if (y != -100).any() else 1]
    part = lce_rows(H, W, y, lse, trows, vrows)
    assert np.allclose(part["dH"], full["dH"][trows], rtol=1e-11, atol=1e-14)
    assert np.allclose(part["dH_abs"], full["dH_abs"][trows], rtol=1e-11, atol=1e-14)
    assert np.allclose(part["dW"], full["dW"][vrows], rtol=1e-11, atol=1e-14)
    assert np.allclose(part["dW_abs"], full["dW_abs"][vrows], rtol=1e-11, atol=1e-14)

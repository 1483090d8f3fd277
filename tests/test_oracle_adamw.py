"""Pins for the fp64 AdamW oracle and its bf16 rounding (CPU only).

Each test ties the oracle to something other than itself: a hand-derived
table, a closed form of Adam's recurrence, an invariant, or the library
AdamW of torch run in float64.
"""

import os

import numpy as np
import pytest
import torch

from oracle import adamw as oa
from oracle import bf16 as ob

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
HP = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


# ---------------------------------------------------------------- bf16 ----

def test_bf16_golden_table():
    for hexval, bits, *_ in _rows("bf16_rne.txt"):
        x = float.fromhex(hexval)
        got = int(ob.bf16_bits(np.array([x]))[0])
        assert got == int(bits, 16), (hexval, hex(got), bits)


def test_bf16_matches_torch_on_fp32_inputs():
    # For inputs that are fp32 values, torch's fp32 -> bf16 conversion is a
    # library RNE; the oracle rounds from fp64 and must agree bit for bit.
    rng = np.random.default_rng(1)
    x32 = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(0.02),
        rng.standard_normal(20000).astype(np.float32) * np.float32(1e30),
        rng.standard_normal(20000).astype(np.float32) * np.float32(1e-39),
        (rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32)).view(np.float32),
    ])
    x32 = x32[np.isfinite(x32)]
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = ob.bf16_bits(x32.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_ulp_distance():
    a = ob.bf16_bits(np.array([1.0, -0.0, 0.0, 2.0 ** -133]))
    b = ob.bf16_bits(np.array([1.0 + 2 ** -7, 0.0, -(2.0 ** -133), -(2.0 ** -133)]))
    assert list(ob.ulp_distance(a, b)) == [1, 0, 1, 2]


# ------------------------------------------------------- bias corrections --

def test_bias_corrections_golden():
    for t, bc1, bc2 in _rows("bias_corrections.txt"):
        g1, g2 = oa.bias_corrections(int(t), 0.9, 0.999)
        assert g1 == pytest.approx(float(bc1), rel=1e-14)
        assert g2 == pytest.approx(float(bc2), rel=1e-12)


def test_bias_corrections_reject_step0():
    with pytest.raises(ValueError):
        oa.bias_corrections(0, 0.9, 0.999)


# ------------------------------------------------------------ closed forms --

def _state(n=4096, seed=0):
    rng = np.random.default_rng(seed)
    th = rng.standard_normal(n) * 0.02
    g = rng.standard_normal(n) * 1e-3
    g[:5] = [0.0, 1e-12, -1e-12, 5.0, -5.0]
    return th, g


def test_first_step_closed_form():
    # At t=1: m_hat = g and v_hat = g**2, so the step is g / (|g| + eps).
    th, g = _state()
    st = oa.AdamWState(th)
    oa.adamw_step(st, g, 1, **HP)
    lam = HP["lr"] * HP["weight_decay"]
    want = th * (1 - lam) - HP["lr"] * g / (np.abs(g) + HP["eps"])
    np.testing.assert_allclose(st.theta, want, rtol=1e-13, atol=1e-18)
    np.testing.assert_allclose(st.m, 0.1 * g, rtol=1e-13, atol=0)
    np.testing.assert_allclose(st.v, 1e-3 * g * g, rtol=1e-12, atol=0)


@pytest.mark.parametrize("t_max", [3, 22])
def test_constant_gradient_closed_form(t_max):
    # With a constant gradient m_hat = g and v_hat = g**2 at every step, so
    # theta_t = (1-lam)**t theta0 - lr*s*(1-(1-lam)**t)/lam, s = g/(|g|+eps).
    th, g = _state(seed=3)
    st = oa.AdamWState(th)
    lam = HP["lr"] * HP["weight_decay"]
    s = g / (np.abs(g) + HP["eps"])
    for t in range(1, t_max + 1):
        oa.adamw_step(st, g, t, **HP)
        geo = -np.expm1(t * np.log1p(-lam)) / lam     # (1-(1-lam)**t)/lam, no cancellation
        want = (1 - lam) ** t * th - HP["lr"] * s * geo
        np.testing.assert_allclose(st.theta, want, rtol=1e-11, atol=1e-17)
        np.testing.assert_allclose(st.m, (1 - 0.9 ** t) * g, rtol=1e-12, atol=0)
        np.testing.assert_allclose(st.v, (1 - 0.999 ** t) * g * g, rtol=1e-10, atol=0)


def test_zero_gradient_only_decays():
    th, _ = _state()
    st = oa.AdamWState(th)
    for t in (1, 2, 3):
        oa.adamw_step(st, np.zeros_like(th), t, **HP)
    assert np.all(st.m == 0) and np.all(st.v == 0)
    np.testing.assert_allclose(st.theta, th * (1 - 1e-6) ** 3, rtol=1e-14)


def test_alternating_sign_second_step():
    # g1 = +h, g2 = -h: m2 = -(1-b1)**2 h, v2 = (1-b2)(1+b2) h**2.
    th, g = _state(seed=5)
    st = oa.AdamWState(th)
    oa.adamw_step(st, g, 1, **HP)
    oa.adamw_step(st, -g, 2, **HP)
    np.testing.assert_allclose(st.m, -(0.1 ** 2) * g, rtol=1e-12)
    np.testing.assert_allclose(st.v, 0.001 * 1.999 * g * g, rtol=1e-12)


def test_scale_invariance_without_eps():
    # Adam's step is invariant to a positive rescaling of all gradients when eps = 0.
    th, g = _state(seed=7)
    g[:3] = [1e-3, -2e-3, 3e-4]
    hp = dict(HP, eps=0.0)
    a, b = oa.AdamWState(th), oa.AdamWState(th)
    rng = np.random.default_rng(8)
    for t in (1, 2, 3):
        gt = g * rng.uniform(0.5, 2.0, g.size)
        oa.adamw_step(a, gt, t, **hp)
        oa.adamw_step(b, 37.0 * gt, t, **hp)
    np.testing.assert_allclose(a.theta, b.theta, rtol=1e-13)


def test_matches_torch_adamw_float64():
    # torch.optim.AdamW (non-amsgrad) is the library form of the same
    # published algorithm; run it in float64 with changing gradients.
    rng = np.random.default_rng(11)
    th = rng.standard_normal(3000) * 0.02
    p = torch.nn.Parameter(torch.from_numpy(th.copy()))
    opt = torch.optim.AdamW([p], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]),
                            eps=HP["eps"], weight_decay=HP["weight_decay"], foreach=False)
    st = oa.AdamWState(th)
    for t in range(1, 6):
        g = rng.standard_normal(th.size) * 10.0 ** rng.uniform(-6, 0, th.size)
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        oa.adamw_step(st, g, t, **HP)
        # theta may cancel (decay vs step): bound the error by its term magnitude
        assert np.all(np.abs(st.theta - p.detach().numpy()) <= 1e-13 * st.theta_abs)
        sd = opt.state[p]
        assert np.all(np.abs(st.m - sd["exp_avg"].numpy()) <= 1e-13 * st.m_abs)
        np.testing.assert_allclose(st.v, sd["exp_avg_sq"].numpy(), rtol=1e-13, atol=0)


def test_weights_are_rne_of_theta():
    th, g = _state(seed=9)
    st = oa.AdamWState(th)
    bits = oa.adamw_step(st, g, 1, **HP)
    want = torch.from_numpy(st.theta.astype(np.float32)).to(torch.bfloat16)
    got = ob.bits_to_f64(bits)
    # theta rounded straight to bf16 vs via fp32: at most one step apart.
    assert np.max(ob.ulp_distance(bits, want.view(torch.int16).numpy().view(np.uint16))) <= 1
    assert np.all(np.abs(got - st.theta) <= np.abs(st.theta) * 2.0 ** -8)


def test_magnitudes_bound_terms():
    th, g = _state(seed=10)
    st = oa.AdamWState(th)
    for t in (1, 2, 3):
        oa.adamw_step(st, g * (-1) ** t, t, **HP)
        assert np.all(st.m_abs >= np.abs(st.m) * (1 - 1e-15))
        assert np.all(st.theta_abs >= np.abs(st.theta) * (1 - 1e-15))


def test_compressed_step_first_step_closed_form():
    rng = np.random.default_rng(12)
    S = rng.standard_normal((16, 16)) * 1e-3
    dS, m, v, dS_abs, _ = oa.compressed_adamw_step(S, np.zeros_like(S), np.zeros_like(S), 1,
                                                   HP["lr"], HP["beta1"], HP["beta2"], HP["eps"])
    np.testing.assert_allclose(dS, HP["lr"] * S / (np.abs(S) + HP["eps"]), rtol=1e-13)
    np.testing.assert_allclose(np.abs(dS), dS_abs, rtol=1e-13)


def test_compressed_step_is_adamw_without_decay():
    # With weight decay 0 and theta = 0, theta_t = -(sum of the steps), which
    # the compressed step returns one by one.
    rng = np.random.default_rng(13)
    S = [rng.standard_normal(64) * 1e-3 for _ in range(3)]
    st = oa.AdamWState(np.zeros(64))
    m = v = np.zeros(64)
    acc = np.zeros(64)
    for t in (1, 2, 3):
        oa.adamw_step(st, S[t - 1], t, **dict(HP, weight_decay=0.0))
        dS, m, v, _, _ = oa.compressed_adamw_step(S[t - 1], m, v, t, HP["lr"], HP["beta1"],
                                                  HP["beta2"], HP["eps"])
        acc -= dS
        np.testing.assert_allclose(acc, st.theta, rtol=1e-13, atol=1e-20)

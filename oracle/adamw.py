"""fp64 AdamW layer step (test infrastructure only).

What it follows
---------------
The layer-sliding engine of "An Efficient Heterogeneous Co-Design for
Fine-Tuning on a Single GPU" updates one layer at a time with Adam on
flattened fp32 optimizer states and writes the low-precision weights back
(technical summary, section 2.A "asynchronous update", section 2.B "shared
buffers for gradients and type conversion", "flattened optimizer states").
The pages name Adam but print no formula, so the update written out here is
the published one: Adam with bias-corrected moments (Kingma & Ba 2015,
Algorithm 1) and decoupled weight decay (Loshchilov & Hutter 2019,
Algorithm 2, "AdamW"), in the order of torch.optim.AdamW without amsgrad:

    theta <- theta * (1 - lr * wd)
    m     <- beta1 * m + (1 - beta1) * g
    v     <- beta2 * v + (1 - beta2) * g**2
    m_hat  = m / (1 - beta1**t)
    v_hat  = v / (1 - beta2**t)
    theta <- theta - lr * m_hat / (sqrt(v_hat) + eps)
    w      = RNE_bf16(theta)

For the compressed space of the learned-sparse-projector path the same
moment update runs on S, with no weight decay (there is no compressed
weight to decay), and the result is the step itself:

    dS = lr * m_hat / (sqrt(v_hat) + eps)

Every quantity also carries an "absolute-term magnitude": the same
expression with every term replaced by its absolute value.  It bounds the
size of the rounding error an fp32 implementation can make, where plain
relative error is meaningless because terms cancel (m at t=2 is
0.09*g1 + 0.1*g2).
"""

import numpy as np

from .bf16 import bf16_bits


def bias_corrections(t, beta1, beta2):
    """(1 - beta1**t, 1 - beta2**t) for step t >= 1, in float64."""
    if t < 1:
        raise ValueError("step t must be >= 1")
    return 1.0 - beta1 ** t, 1.0 - beta2 ** t


class AdamWState:
    """Per-element fp64 state of one tensor: theta, m, v and their magnitudes."""

    def __init__(self, theta, m=None, v=None):
        theta = np.asarray(theta, dtype=np.float64)
        self.theta = theta.copy()
        self.m = np.zeros_like(theta) if m is None else np.asarray(m, np.float64).copy()
        self.v = np.zeros_like(theta) if v is None else np.asarray(v, np.float64).copy()
        self.theta_abs = np.abs(self.theta)
        self.m_abs = np.abs(self.m)
        self.v_abs = np.abs(self.v)


def adamw_step(state, g, t, lr, beta1, beta2, eps, weight_decay):
    """One AdamW step on ``state`` (in place) with gradient ``g`` at step ``t``.

    Returns the bf16 bit pattern of the new weights.
    """
    g = np.asarray(g, dtype=np.float64)
    bc1, bc2 = bias_corrections(t, beta1, beta2)
    decay = 1.0 - lr * weight_decay

    m = beta1 * state.m + (1.0 - beta1) * g
    v = beta2 * state.v + (1.0 - beta2) * g * g
    m_hat = m / bc1
    v_hat = v / bc2
    update = lr * m_hat / (np.sqrt(v_hat) + eps)
    theta = state.theta * decay - update

    m_abs = beta1 * state.m_abs + (1.0 - beta1) * np.abs(g)
    v_abs = beta2 * state.v_abs + (1.0 - beta2) * g * g
    upd_abs = lr * (m_abs / bc1) / (np.sqrt(v / bc2) + eps)
    theta_abs = state.theta_abs * abs(decay) + upd_abs

    state.theta, state.m, state.v = theta, m, v
    state.theta_abs, state.m_abs, state.v_abs = theta_abs, m_abs, v_abs
    return bf16_bits(theta)


def compressed_adamw_step(S, m, v, t, lr, beta1, beta2, eps, m_abs=None):
    """AdamW moments on the compressed gradient S.

    No weight decay: the compressed space holds no weight.  ``m`` and ``v``
    are the previous fp64 moments (zeros before the first step) and
    ``m_abs`` the previous magnitude of m (defaults to |m|).  Returns
    ``(dS, m_new, v_new, dS_abs, m_abs_new)``.
    """
    S = np.asarray(S, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m_abs = np.abs(m) if m_abs is None else np.asarray(m_abs, np.float64)
    bc1, bc2 = bias_corrections(t, beta1, beta2)
    m_new = beta1 * m + (1.0 - beta1) * S
    v_new = beta2 * v + (1.0 - beta2) * S * S
    dS = lr * (m_new / bc1) / (np.sqrt(v_new / bc2) + eps)
    m_abs_new = beta1 * m_abs + (1.0 - beta1) * np.abs(S)
    dS_abs = lr * (m_abs_new / bc1) / (np.sqrt(v_new / bc2) + eps)
    return dS, m_new, v_new, dS_abs, m_abs_new

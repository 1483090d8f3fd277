"""fp64 projector fit step (test infrastructure only).

What it follows
---------------
"Practical offloading for fine-tuning LLM on commodity GPU via learned
sparse projectors" (LSP-Offload; abstract, and the method section's "key
design" paragraph): the sparse projectors are learned from data by a
gradient-descent method whose objective is the precision lost by
compressing and then decompressing.  The pages give neither the loss nor
the schedule; the plainest reading, used here, is one plain gradient step
on the stored nonzero values of P and Q (their column ids stay fixed) for
the squared Frobenius reconstruction error of a gradient sample G:

    S = P^T G Q,   R = P S Q^T,   E = G - R,   L = ||E||_F^2

    dL/dP = -2 (E Q S^T + G Q Q^T E^T P)          (m x d, dense)
    dL/dQ = -2 (E^T P S + G^T P P^T E Q)          (n x d, dense)

and the gradient of a stored value is the dense gradient at its (row, id)
position (a repeated id in a row adds up in P, so both copies see the same
gradient).  The step is  val <- val - lr * grad  for P and Q at once, both
gradients taken at the values before the step.

Every product is numpy matmul on dense fp64 copies: the definition written
out, one library primitive per product.  Alongside each quantity the oracle
returns its absolute-term magnitude (the same expression with every factor
replaced by the magnitude of its terms), which bounds the rounding error of
an fp32 evaluation in any summation order.
"""

import numpy as np

from .lsp import Projector


def fit_loss(G, P, Q):
    """||G - P P^T G Q Q^T||_F^2 in fp64."""
    G = np.asarray(G, dtype=np.float64)
    Pd, Qd = P.dense(), Q.dense()
    S = Pd.T @ G @ Qd
    E = G - Pd @ S @ Qd.T
    return float(np.sum(E * E))


def fit_step(G, P, Q, lr):
    """One gradient step on the values of P and Q.

    Returns a dict with
      loss, loss_abs        L before the step and its term magnitude
      gP, gQ                gradients per stored value, [rows, k] (ELL order)
      gP_abs, gQ_abs        their term magnitudes
      P_val, Q_val          values after the step, [rows, k]
    """
    G = np.asarray(G, dtype=np.float64)
    Pd, Qd = P.dense(), Q.dense()
    aG, aP, aQ = np.abs(G), np.abs(Pd), np.abs(Qd)

    S = Pd.T @ G @ Qd
    R = Pd @ S @ Qd.T
    E = G - R
    S_abs = aP.T @ aG @ aQ
    R_abs = aP @ S_abs @ aQ.T
    E_abs = aG + R_abs

    gPd = -2.0 * (E @ Qd @ S.T + G @ Qd @ Qd.T @ E.T @ Pd)
    gQd = -2.0 * (E.T @ Pd @ S + G.T @ Pd @ Pd.T @ E @ Qd)
    gPd_abs = 2.0 * (E_abs @ aQ @ S_abs.T + aG @ aQ @ aQ.T @ E_abs.T @ aP)
    gQd_abs = 2.0 * (E_abs.T @ aP @ S_abs + aG.T @ aP @ aP.T @ E_abs @ aQ)

    rP = np.repeat(np.arange(P.rows), P.k).reshape(P.rows, P.k)
    rQ = np.repeat(np.arange(Q.rows), Q.k).reshape(Q.rows, Q.k)
    gP, gQ = gPd[rP, P.idx], gQd[rQ, Q.idx]
    out = {
        "loss": float(np.sum(E * E)),
        "loss_abs": float(np.sum(aG * aG) + 2.0 * np.sum(aG * R_abs) + np.sum(R_abs * R_abs)),
        "gP": gP,
        "gQ": gQ,
        "gP_abs": gPd_abs[rP, P.idx],
        "gQ_abs": gQd_abs[rQ, Q.idx],
        "P_val": P.val - lr * gP,
        "Q_val": Q.val - lr * gQ,
    }
    return out


def stepped(P, Q, res):
    """The projectors after a step, as new Projector objects."""
    return Projector(P.idx, res["P_val"], P.d), Projector(Q.idx, res["Q_val"], Q.d)

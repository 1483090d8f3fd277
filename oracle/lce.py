"""fp64 linear cross-entropy (test infrastructure only).

What it follows
---------------
SlideFormer ("An Efficient Heterogeneous Co-Design for Fine-Tuning on a
Single GPU"; the German summary's kernel list, the Spanish summary's
"Kernel Fused LinearCrossEntropy", the French summary's "Noyaux Triton
optimises"): the output projection and the loss are fused, and the
gradients are computed in small blocks so that the full logits tensor is
never held.  The pages give no formula; the operation is the standard
softmax cross-entropy of a linear output layer, averaged over the tokens
that carry a label:

    z_i  = W h_i                        (V logits of token i)
    L    = (1/n) sum_{i labelled} ( logsumexp(z_i) - z_i[y_i] )
    dZ_i = (softmax(z_i) - onehot(y_i)) / n    (0 for unlabelled tokens)
    dH   = dZ W,   dW = dZ^T H

with n the number of labelled tokens (label != ignore_index).  Everything
is fp64 numpy on the exact input values; alongside dH and dW the oracle
returns their absolute-term magnitudes |dZ| |W| and |dZ|^T |H|.
"""

import numpy as np


def lce(H, W, labels, ignore_index=-100):
    """Loss, dH, dW and magnitudes for hidden states H [N, D], weight W [V, D]."""
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    y = np.asarray(labels, dtype=np.int64)
    N, V = H.shape[0], W.shape[0]
    valid = y != ignore_index
    n = int(valid.sum())
    Z = H @ W.T
    zmax = Z.max(axis=1, keepdims=True)
    lse = (zmax + np.log(np.exp(Z - zmax).sum(axis=1, keepdims=True)))[:, 0]
    P = np.exp(Z - lse[:, None])
    dZ = np.zeros_like(Z)
    loss = 0.0
    if n:
        rows = np.flatnonzero(valid)
        loss = float(np.sum(lse[rows] - Z[rows, y[rows]]) / n)
        dZ[rows] = P[rows]
        dZ[rows, y[rows]] -= 1.0
        dZ /= n
    aZ = np.abs(dZ)
    return {
        "loss": loss,
        "lse": lse,
        "Z": Z,
        "dZ": dZ,
        "dH": dZ @ W,
        "dW": dZ.T @ H,
        "dH_abs": aZ @ np.abs(W),
        "dW_abs": aZ.T @ np.abs(H),
        "n": n,
    }


def loss_only(H, W, labels, ignore_index=-100):
    """The loss alone (for finite differences)."""
    return lce(H, W, labels, ignore_index)["loss"]

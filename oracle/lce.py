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


def token_lse(H, W, chunk=4096):
    """log sum_v exp(z_iv) for every token, fp64, over the vocabulary in chunks.

    For output layers too large to hold the N x V logits (a Llama-3.1-8B
    head: 8192 x 128256): each chunk of W's rows gives a block of logits,
    folded into a running maximum and a running sum of exponentials
    rescaled to it, so the result is the log-sum-exp of the whole row up to
    fp64 rounding.
    """
    H = np.asarray(H, dtype=np.float64)
    N, V = H.shape[0], W.shape[0]
    m = np.full(N, -np.inf)
    s = np.zeros(N)
    for v0 in range(0, V, chunk):
        Z = H @ np.asarray(W[v0:v0 + chunk], dtype=np.float64).T
        mn = np.maximum(m, Z.max(axis=1))
        s = s * np.exp(m - mn) + np.exp(Z - mn[:, None]).sum(axis=1)
        m = mn
    return m + np.log(s)


def lce_rows(H, W, labels, lse, token_rows, vocab_rows, ignore_index=-100):
    """Selected rows of dH and dW (with magnitudes) given every token's lse.

    dH[i] = sum_v dZ[i, v] W[v] needs token i's whole row of dZ; dW[v] =
    sum_i dZ[i, v] H[i] needs column v of dZ for every token, which the
    per-token log-sum-exp gives without the other logits:
    dZ[i, v] = (exp(z_iv - lse_i) - [y_i = v]) / n for labelled tokens.
    """
    H = np.asarray(H, dtype=np.float64)
    y = np.asarray(labels, dtype=np.int64)
    valid = y != ignore_index
    n = int(valid.sum())
    token_rows = np.asarray(token_rows, dtype=np.int64)
    vocab_rows = np.asarray(vocab_rows, dtype=np.int64)
    W = np.asarray(W)
    dH = np.zeros((len(token_rows), H.shape[1]))
    dH_abs = np.zeros_like(dH)
    V = W.shape[0]
    for v0 in range(0, V, 8192):
        Wc = np.asarray(W[v0:v0 + 8192], dtype=np.float64)
        Zr = H[token_rows] @ Wc.T
        dZr = np.exp(Zr - lse[token_rows][:, None])
        for r, i in enumerate(token_rows):
            if valid[i] and v0 <= y[i] < v0 + Wc.shape[0]:
                dZr[r, y[i] - v0] -= 1.0
        dZr = np.where(valid[token_rows][:, None], dZr / max(n, 1), 0.0)
        dH += dZr @ Wc
        dH_abs += np.abs(dZr) @ np.abs(Wc)
    Wv = np.asarray(W[vocab_rows], dtype=np.float64)
    Zc = H @ Wv.T                                      # [N, len(vocab_rows)]
    dZc = np.exp(Zc - lse[:, None])
    onehot = y[:, None] == vocab_rows[None, :]
    dZc = np.where(valid[:, None], (dZc - onehot) / max(n, 1), 0.0)
    return {"dH": dH, "dH_abs": dH_abs, "dW": dZc.T @ H, "dW_abs": np.abs(dZc).T @ np.abs(H), "n": n}

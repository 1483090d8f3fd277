"""Projector fit step against the fp64 oracle (GPU).

One gradient step on the stored values of P and Q for the reconstruction
error ||G - P P^T G Q Q^T||_F^2: the loss, both gradients (in ELL order),
the stepped values, and that compress / decompress-apply afterwards use the
new values in every layout the library keeps.
"""

import numpy as np
import pytest
import torch

from _util import TOL_LSP, check_close, f64
from layer_optimizer_gb300 import native, synth
from oracle import lsp as ol
from oracle import lsp_fit as of

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _make(rows, d, k, seed):
    idx, val = synth.projector(rows, d, k, seed)
    h = native.lsp_projector_create(rows, d, k, torch.from_numpy(idx).to(DEV), torch.from_numpy(val).to(DEV))
    return h, ol.Projector(idx, val, d)


def _fit(P, Q, G, g_dtype, m, n, d, lr):
    wsb = native.lsp_fit_workspace_bytes(m, n, d, g_dtype)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    loss = torch.full((1,), float("nan"), dtype=torch.float64, device=DEV)
    gP = torch.empty(m * P.k, device=DEV)
    gQ = torch.empty(n * Q.k, device=DEV)
    native.lsp_projector_fit_step(P, Q, G, g_dtype, m, n, lr, loss, gP, gQ, ws, wsb)
    torch.cuda.synchronize()
    return float(loss.item()), gP.view(m, P.k), gQ.view(n, Q.k)


def _values(h, rows, k):
    v = torch.empty(rows * k, device=DEV)
    native.lsp_projector_export_values(h, v)
    torch.cuda.synchronize()
    return v.view(rows, k)


def _gradient(m, n, g_dtype, seed):
    G = synth.normal((m, n), 1e-3, seed, dtype=torch.bfloat16 if g_dtype == native.SF_BF16 else torch.float32)
    return G.to(DEV), f64(G)


@pytest.mark.parametrize("m,n,d,k,g_dtype", [
    (300, 200, 64, 4, native.SF_FP32),
    (256, 384, 32, 2, native.SF_BF16),
    (130, 264, 96, 3, native.SF_FP32),      # rows not a multiple of 4: generic gather for G Q
    (1024, 1024, 64, 4, native.SF_BF16),    # the one-linear-layer projector shape
    (640, 520, 128, 5, native.SF_FP32),     # d x d products split over clusters, one slab per part
    (384, 1000, 256, 8, native.SF_BF16),    # rows of G^T Q in 16-byte pieces, k = 8
    (4096, 4096, 512, 8, native.SF_FP32),   # a LLaMA-7B attention matrix
])
def test_fit_step_matches_oracle(m, n, d, k, g_dtype):
    hP, P = _make(m, d, k, 31 + m)
    hQ, Q = _make(n, d, k, 47 + n)
    G, G64 = _gradient(m, n, g_dtype, 5 + m + n)
    lr = 1e-3
    loss, gP, gQ = _fit(hP, hQ, G, g_dtype, m, n, d, lr)
    ref = of.fit_step(G64, P, Q, lr)

    assert abs(loss - ref["loss"]) <= TOL_LSP * ref["loss_abs"], (loss, ref["loss"], ref["loss_abs"])
    check_close("dL/dP", gP, ref["gP"], ref["gP_abs"], TOL_LSP)
    check_close("dL/dQ", gQ, ref["gQ"], ref["gQ_abs"], TOL_LSP)

    # the step: every stored value moved by -lr * (its own gradient), in fp32
    vP, vQ = _values(hP, m, k), _values(hQ, n, k)
    lr32 = float(np.float32(lr))
    for v_new, v_old, g in ((vP, P.val, gP), (vQ, Q.val, gQ)):
        v0, gg = v_old.astype(np.float32).astype(np.float64), f64(g)
        err = np.abs(f64(v_new) - (v0 - lr32 * gg))          # one fp32 rounding of the exact step
        assert np.all(err <= 2.0 ** -24 * np.abs(v0 - lr32 * gg) * 1.0001 + 1e-45)
    check_close("P values", vP, ref["P_val"], np.abs(P.val) + lr * ref["gP_abs"], TOL_LSP)
    check_close("Q values", vQ, ref["Q_val"], np.abs(Q.val) + lr * ref["gQ_abs"], TOL_LSP)

    # compress afterwards uses the new values (CSC and window-major copies)
    P2, Q2 = ol.Projector(P.idx, f64(vP), d), ol.Projector(Q.idx, f64(vQ), d)
    wsb = native.lsp_workspace_bytes(m, n, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    S = torch.empty(d, d, device=DEV)
    native.lsp_compress(hP, hQ, G, g_dtype, m, n, S, ws, wsb)
    # ... and decompress-apply (the ELL copies) on an fp32 W of zeros gives -P dS Q^T
    dS = synth.normal((d, d), 1e-4, 77).to(DEV)
    W = torch.zeros(m, n, device=DEV)
    native.lsp_decompress_apply(hP, hQ, dS, W, native.SF_FP32, None, m, n, ws, wsb)
    torch.cuda.synchronize()
    S_ref, S_abs = ol.compress(P2, Q2, G64)
    check_close("S after the step", S, S_ref, S_abs, TOL_LSP)
    D, D_abs = ol.decompress(P2, Q2, f64(dS))
    check_close("apply after the step", W, -D, D_abs, TOL_LSP)


@pytest.mark.parametrize("k", [4, 40])
def test_fit_step_with_repeated_ids(k):
    # projectors built without validation may repeat an id inside a row (the
    # values then add up); k = 40 also takes the Gram matrices' multi-pass path
    m, n, d = 300, 200, 64
    hPQ = []
    for rows, seed in ((m, 131), (n, 137)):
        idx, val = synth.projector(rows, d, k, seed)
        idx[::7, 1] = idx[::7, 0]                 # every 7th row repeats its first id
        idx[::11, k - 1] = idx[::11, 1]
        h = native.lsp_projector_create(rows, d, k, torch.from_numpy(idx).to(DEV), torch.from_numpy(val).to(DEV),
                                        validate=False)
        hPQ.append((h, ol.Projector(idx, val, d)))
    (hP, P), (hQ, Q) = hPQ
    G, G64 = _gradient(m, n, native.SF_FP32, 141)
    loss, gP, gQ = _fit(hP, hQ, G, native.SF_FP32, m, n, d, 1e-3)
    ref = of.fit_step(G64, P, Q, 1e-3)
    assert abs(loss - ref["loss"]) <= TOL_LSP * ref["loss_abs"], (loss, ref["loss"], ref["loss_abs"])
    check_close("dL/dP", gP, ref["gP"], ref["gP_abs"], TOL_LSP)
    check_close("dL/dQ", gQ, ref["gQ"], ref["gQ_abs"], TOL_LSP)


def test_fit_steps_descend_and_are_deterministic():
    m, n, d, k = 512, 384, 64, 4
    hP, P = _make(m, d, k, 3)
    hQ, Q = _make(n, d, k, 4)
    G, G64 = _gradient(m, n, native.SF_FP32, 9)
    loss0, gP, gQ = _fit(hP, hQ, G, native.SF_FP32, m, n, d, 0.0)
    # lr = 0 evaluates only: the values stay as created
    assert np.array_equal(f64(_values(hP, m, k)), P.val.astype(np.float32).astype(np.float64))
    # the same call twice gives the same bits
    loss0b, gPb, gQb = _fit(hP, hQ, G, native.SF_FP32, m, n, d, 0.0)
    assert loss0 == loss0b and torch.equal(gP, gPb) and torch.equal(gQ, gQb)
    g2 = float((gP.double() ** 2).sum() + (gQ.double() ** 2).sum())
    lr = 0.05 * loss0 / g2
    # each call reports the loss before its own step
    losses = [_fit(hP, hQ, G, native.SF_FP32, m, n, d, lr)[0] for _ in range(4)]
    final = _fit(hP, hQ, G, native.SF_FP32, m, n, d, 0.0)[0]
    losses.append(final)
    assert losses[0] == loss0
    assert all(b < a for a, b in zip(losses, losses[1:])), losses
    # the loss the library reports after the steps is the oracle's for the values it holds
    P2 = ol.Projector(P.idx, f64(_values(hP, m, k)), d)
    Q2 = ol.Projector(Q.idx, f64(_values(hQ, n, k)), d)
    ref = of.fit_step(G64, P2, Q2, 0.0)
    assert abs(final - ref["loss"]) <= TOL_LSP * ref["loss_abs"]


def test_fit_rejects_bad_arguments():
    m, n, d, k = 64, 48, 16, 2
    hP, _ = _make(m, d, k, 1)
    hQ, _ = _make(n, d, k, 2)
    G, _ = _gradient(m, n, native.SF_FP32, 3)
    wsb = native.lsp_fit_workspace_bytes(m, n, d, native.SF_FP32)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    hS, _ = _make(m, d, k, 5)
    with pytest.raises(native.SfError, match="different"):
        native.lsp_projector_fit_step(hS, hS, torch.zeros(m, m, device=DEV), native.SF_FP32, m, m, 0.1, None, None,
                                      None, ws, wsb)
    with pytest.raises(native.SfError, match="workspace"):
        native.lsp_projector_fit_step(hP, hQ, G, native.SF_FP32, m, n, 0.1, None, None, None, ws, 256)
    with pytest.raises(native.SfError, match="finite"):
        native.lsp_projector_fit_step(hP, hQ, G, native.SF_FP32, m, n, float("nan"), None, None, None, ws, wsb)
    with pytest.raises(native.SfError, match="rows"):
        native.lsp_projector_fit_step(hQ, hP, G, native.SF_FP32, m, n, 0.1, None, None, None, ws, wsb)
    idx, val = synth.projector(m, d, k, 6)
    idx[3, 0] = d + 5                                   # out of range, accepted unvalidated
    hB = native.lsp_projector_create(m, d, k, torch.from_numpy(idx).to(DEV), torch.from_numpy(val).to(DEV),
                                     validate=False)
    with pytest.raises(native.SfError, match="outside"):
        native.lsp_projector_fit_step(hB, hQ, G, native.SF_FP32, m, n, 0.1, None, None, None, ws, wsb)

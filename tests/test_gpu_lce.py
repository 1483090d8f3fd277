"""Fused linear cross-entropy against the fp64 oracle (GPU).

Tolerances: the logits are bf16 products summed in fp32, so the loss is
checked to 1e-5 of the logit magnitude sum |h||w|; dZ is rounded to bf16
before the gradient products (relative error <= 2^-9 per entry), so dH and
dW are checked to 2^-8 of their absolute-term magnitudes |dZ||W| and
|dZ|^T|H|.
"""

import numpy as np
import pytest
import torch

from _util import check_close, f64
from layer_optimizer_gb300 import native, synth
from oracle.lce import lce

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_GRAD = 2.0 ** -8


def _case(N, D, V, seed, n_ignore=0):
    H = synth.normal((N, D), 1.0, seed, dtype=torch.bfloat16)
    W = synth.normal((V, D), 0.02, seed + 1, dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(seed + 2)
    y = torch.randint(0, V, (N,), generator=g, dtype=torch.int32)
    if n_ignore:
        y[torch.randperm(N, generator=g)[:n_ignore]] = -100
    return H, W, y


def _run(H, W, y, chunk, grads=True):
    N, D = H.shape
    V = W.shape[0]
    wsb = native.lce_workspace_bytes(N, D, V, chunk)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    loss = torch.full((1,), float("nan"), dtype=torch.float64, device=DEV)
    dH = torch.full((N, D), float("nan"), device=DEV) if grads else None
    dW = torch.full((V, D), float("nan"), device=DEV) if grads else None
    native.lce_forward_backward(H.to(DEV), W.to(DEV), y.to(DEV), N, D, V, chunk, -100, loss, dH, dW, ws, wsb)
    torch.cuda.synchronize()
    native.sf_sync_status()
    return loss.item(), dH, dW


def _check(res, loss, dH, dW, H64, W64):
    Z_abs = np.abs(H64) @ np.abs(W64).T
    labelled = res["n"]
    if labelled:
        bound = 1e-5 * Z_abs.max(axis=1).mean() * 2 + 1e-6 * np.abs(res["lse"]).mean()
        assert abs(loss - res["loss"]) <= bound, (loss, res["loss"], bound)
    else:
        assert loss == 0.0
    for name, got, ref, mag in (("dH", dH, res["dH"], res["dH_abs"]), ("dW", dW, res["dW"], res["dW_abs"])):
        err = np.abs(f64(got) - ref)
        bad = err > TOL_GRAD * mag + 1e-30
        assert not bad.any(), (name, int(bad.sum()), float((err / (mag + 1e-30)).max()))


@pytest.mark.parametrize("N,D,V,chunk,n_ignore", [
    (300, 64, 520, 128, 20),
    (1000, 256, 1000, 256, 0),
    (64, 8, 8, 64, 5),
    (130, 96, 2048, 64, 1),       # ragged last chunk
    (40, 32, 264, 512, 40),       # every token unlabelled
])
def test_lce_matches_oracle(N, D, V, chunk, n_ignore):
    H, W, y = _case(N, D, V, N + D + V, n_ignore)
    loss, dH, dW = _run(H, W, y, chunk)
    H64, W64 = f64(H), f64(W)
    res = lce(H64, W64, y.numpy())
    _check(res, loss, dH, dW, H64, W64)


def test_lce_llama_head_shape():
    # a LLaMA-2-7B output layer (V 32000, D 4096) on 2048 tokens in two chunks
    N, D, V = 2048, 4096, 32000
    H, W, y = _case(N, D, V, 17, 64)
    loss, dH, dW = _run(H, W, y, 1024)
    H64, W64 = f64(H), f64(W)
    _check(lce(H64, W64, y.numpy()), loss, dH, dW, H64, W64)


def test_lce_chunking_loss_only_and_determinism():
    N, D, V = 500, 128, 1024
    H, W, y = _case(N, D, V, 23, 30)
    l1, dH1, dW1 = _run(H, W, y, 64)
    l2, dH2, dW2 = _run(H, W, y, 64)
    assert l1 == l2 and torch.equal(dH1, dH2) and torch.equal(dW1, dW2)
    l3, dH3, dW3 = _run(H, W, y, 512)                 # one chunk instead of eight
    assert torch.equal(dH1, dH3)                      # dH rows do not depend on the chunking
    res = lce(f64(H), f64(W), y.numpy())
    _check(res, l3, dH3, dW3, f64(H), f64(W))
    l4, _, _ = _run(H, W, y, 256, grads=False)
    assert abs(l4 - l1) <= 1e-6 * abs(l1)


def test_lce_rejects_and_flags():
    N, D, V = 64, 16, 64
    H, W, y = _case(N, D, V, 5)
    ws = torch.empty(native.lce_workspace_bytes(N, D, V, 64), dtype=torch.uint8, device=DEV)
    loss = torch.empty(1, dtype=torch.float64, device=DEV)
    with pytest.raises(native.SfError, match="multiple of 8"):
        native.lce_forward_backward(H.to(DEV), W.to(DEV), y.to(DEV), N, D, V, 60, -100, loss, None, None, ws,
                                    ws.numel())
    with pytest.raises(native.SfError, match="workspace"):
        native.lce_forward_backward(H.to(DEV), W.to(DEV), y.to(DEV), N, D, V, 64, -100, loss, None, None, ws, 256)
    Hb = torch.zeros(N, 12, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(native.SfError, match="multiples of 8"):
        native.lce_forward_backward(Hb, W.to(DEV), y.to(DEV), N, 12, V, 64, -100, loss, None, None, ws, ws.numel())
    y_bad = y.clone()
    y_bad[3] = V + 7                                  # neither a class nor ignore_index
    native.lce_forward_backward(H.to(DEV), W.to(DEV), y_bad.to(DEV), N, D, V, 64, -100, loss, None, None, ws,
                                ws.numel())
    with pytest.raises(native.SfError, match="out-of-range"):
        native.sf_sync_status()


@pytest.mark.slow
def test_lce_llama31_head_full_size_sampled():
    # the benchmark's configuration: 8192 tokens of a Llama-3.1-8B output
    # layer in chunks of 4608.  The oracle takes every token's log-sum-exp
    # in fp64 over vocabulary chunks (the 8192 x 128256 logits are never
    # held), then gives rows of dH (tokens at the chunk edges and an
    # unlabelled one) and rows of dW (vocabulary ids at tile edges and ids
    # that are labels), each compared element by element with the kernels'.
    # dW also keeps a property that holds at any size: every row of dZ sums
    # to zero, so the sum of dW over the vocabulary is zero.
    from oracle.lce import lce_rows, token_lse
    N, D, V, chunk = 8192, 4096, 128256, 4608
    H = synth.fill_normal_(torch.empty(N, D, dtype=torch.bfloat16, device=DEV), 1.0, synth.sub_seed(31, 0))
    W = synth.fill_normal_(torch.empty(V, D, dtype=torch.bfloat16, device=DEV), 0.02, synth.sub_seed(31, 1))
    g = torch.Generator(device=DEV)
    g.manual_seed(synth.sub_seed(31, 2))
    y = torch.randint(0, V, (N,), generator=g, device=DEV, dtype=torch.int32)
    y[::97] = -100
    loss, dH, dW = _run(H, W, y, chunk)
    n = int((y != -100).sum())
    H64, W32, y_np = f64(H), W.float().cpu().numpy(), y.cpu().numpy()
    lse = token_lse(H64, W32, chunk=8192)
    trows = [0, 1, 97, 4607, 4608, 5000, N - 1]
    vrows = [0, 1, 255, 256, 65535, V - 1, int(y_np[3]), int(y_np[4700])]
    ref = lce_rows(H64, W32, y_np, lse, trows, vrows)
    assert ref["n"] == n
    check_close("dH rows", dH[trows], ref["dH"], ref["dH_abs"], TOL_GRAD)
    check_close("dW rows", dW[vrows], ref["dW"], ref["dW_abs"], TOL_GRAD)
    assert not dH[97].any()                               # an unlabelled token has no gradient
    colsum = dW.double().sum(dim=0)
    bound = TOL_GRAD * (2.0 / n) * H.double().abs().sum(dim=0) + 1e-12
    assert bool((colsum.abs() <= bound).all()), float((colsum.abs() / bound).max())
    # the loss from the same log-sum-exps: mean over labelled tokens of lse - z_y,
    # within the bound of the small-size tests with each row's largest |H||W|^T
    # term sum bounded above by |H_i| . max_v |W_v| (no full product needed)
    lab = np.flatnonzero(y_np != -100)
    z_y = np.einsum("ij,ij->i", H64[lab], W32[y_np[lab]].astype(np.float64))
    want = float(np.mean(lse[lab] - z_y))
    row_bound = np.abs(H64) @ np.abs(W32).max(axis=0).astype(np.float64)
    bound = 1e-5 * row_bound.mean() * 2 + 1e-6 * np.abs(lse).mean()
    assert abs(loss - want) <= bound, (loss, want, bound)
    assert 0.0 < loss < 2 * np.log(V)

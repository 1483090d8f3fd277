"""Layer-batched compress (`lsp_compress_layer`) against per-matrix compress and the oracle (GPU).

The layer call runs the first stages of a layer's matrices in one launch and
the second stages in another; every tile is computed as in its own launch,
so S must equal the per-matrix `lsp_compress` results bit for bit.
"""

import pytest
import torch

from _util import TOL_LSP, check_close, f64
from layer_optimizer_gb300 import native, synth
from oracle import lsp as ol

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _proj(rows, d, k, seed):
    idx, val = synth.projector(rows, d, k, seed)
    return native.lsp_projector_create(rows, d, k, torch.from_numpy(idx).to(DEV), torch.from_numpy(val).to(DEV)), \
        ol.Projector(idx, val, d)


def _setup(shapes, d, k, seed):
    mats = []
    for i, (m, n, dt) in enumerate(shapes):
        P, Pr = _proj(m, d, k, seed + 10 * i)
        Q, Qr = _proj(n, d, k, seed + 10 * i + 1)
        G = synth.normal((m, n), 1e-3, seed + 10 * i + 2, dtype=dt).to(DEV)
        g_dtype = native.SF_FP32 if dt == torch.float32 else native.SF_BF16
        mats.append((m, n, P, Q, Pr, Qr, G, g_dtype))
    return mats


def _per_matrix(mats, d):
    out = []
    for (m, n, P, Q, _, _, G, g_dtype) in mats:
        S = torch.full((d, d), float("nan"), device=DEV)
        nb = native.lsp_workspace_bytes(m, n, d)
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=DEV)
        native.lsp_compress(P, Q, G, g_dtype, m, n, S, ws, nb)
        out.append(S)
    torch.cuda.synchronize()
    return out


def _layer(mats, d):
    Ss = [torch.full((d, d), float("nan"), device=DEV) for _ in mats]
    ms, ns = [x[0] for x in mats], [x[1] for x in mats]
    nb = native.lsp_compress_layer_workspace_bytes(ms, ns, d)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    native.lsp_compress_layer([x[2] for x in mats], [x[3] for x in mats], [x[6] for x in mats], [x[7] for x in mats],
                              ms, ns, Ss, ws, nb)
    torch.cuda.synchronize()
    return Ss


def test_layer_compress_equals_per_matrix_bitwise_and_oracle():
    d, k = 512, 8
    shapes = [
        (300, 264, torch.float32),
        (300, 5000, torch.float32),     # past one wave: whole waves plus a split tail
        (520, 136, torch.bfloat16),     # its own launch: the bf16 element type
        (257, 99, torch.float32),       # rows of G not 16-byte multiples: plain-load first stage
        (1024, 1024, torch.float32),
        (130, 2000, torch.bfloat16),
    ]
    mats = _setup(shapes, d, k, 500)
    ref = _per_matrix(mats, d)
    got = _layer(mats, d)
    for i, (a, b) in enumerate(zip(got, ref)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"matrix {i}: not the bits of lsp_compress"
    for i in (1, 2):
        m, n, _, _, Pr, Qr, G, _ = mats[i]
        S_ref, S_abs = ol.compress(Pr, Qr, f64(G.float()))
        check_close(f"S[{i}] vs oracle", got[i], S_ref, S_abs, TOL_LSP)
    native.sf_sync_status()


def test_layer_compress_llama7b_matrices_bitwise():
    d, k = 512, 8
    shapes = [(m, n, torch.float32) for (_, m, n) in synth.LLAMA7_LSP_MATRICES]
    mats = _setup(shapes, d, k, 700)
    ref = _per_matrix(mats, d)
    got = _layer(mats, d)
    for (name, _, _), a, b in zip(synth.LLAMA7_LSP_MATRICES, got, ref):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"{name}: not the bits of lsp_compress"
    native.sf_sync_status()


def test_layer_compress_rejects_bad_arguments():
    d, k = 64, 4
    mats = _setup([(100, 80, torch.float32), (90, 70, torch.float32)], d, k, 900)
    P64, _ = _proj(90, 32, k, 999)                  # a projector of another d
    ms, ns = [100, 90], [80, 70]
    nb = native.lsp_compress_layer_workspace_bytes(ms, ns, d)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    Ss = [torch.empty(d, d, device=DEV) for _ in mats]
    with pytest.raises(native.SfError):             # workspace one byte short
        native.lsp_compress_layer([x[2] for x in mats], [x[3] for x in mats], [x[6] for x in mats],
                                  [native.SF_FP32] * 2, ms, ns, Ss, ws, nb - 1)
    with pytest.raises(native.SfError):             # projectors of different d
        native.lsp_compress_layer([mats[0][2], P64], [mats[0][3], mats[1][3]], [x[6] for x in mats],
                                  [native.SF_FP32] * 2, ms, ns, Ss, ws, nb)
    with pytest.raises(native.SfError):             # rows that do not match m
        native.lsp_compress_layer([x[2] for x in mats], [x[3] for x in mats], [x[6] for x in mats],
                                  [native.SF_FP32] * 2, [100, 91], ns, Ss, ws, nb)
    assert native.lsp_compress_layer_workspace_bytes([], [], d) == 0
    native.sf_sync_status()

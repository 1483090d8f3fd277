"""Seeded sweep of random projector shapes (GPU): compress per matrix against the
oracle, the layer call bit for bit against per-matrix compress, and
decompress-apply against the oracle.

The shapes are drawn so that every launch form of the first stage appears:
small grids with row splits, one wave of whole tiles, grids past one wave
with a split tail, and operands the staged gather cannot take.
"""

import numpy as np
import pytest
import torch

from _util import TOL_LSP, check_close, f64
from layer_optimizer_gb300 import native, synth
from oracle import lsp as ol

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _shapes(seed, count, d):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        m = int(rng.integers(1, 700))
        n = int(rng.choice([rng.integers(1, 300), rng.integers(300, 2000), rng.integers(4800, 6500)]))
        k = int(rng.integers(1, min(16, d) + 1))
        dt = torch.float32 if rng.random() < 0.7 else torch.bfloat16
        out.append((m, n, k, dt))
    return out


def _make(rows, d, k, seed):
    idx, val = synth.projector(rows, d, k, seed)
    return (native.lsp_projector_create(rows, d, k, torch.from_numpy(idx).to(DEV), torch.from_numpy(val).to(DEV)),
            ol.Projector(idx, val, d))


@pytest.mark.parametrize("d,seed", [(8, 1), (64, 2), (200, 3), (512, 4), (1024, 5)])
def test_random_shapes_compress_layer_and_apply(d, seed):
    shapes = _shapes(seed, 6, d)
    mats, per = [], []
    for i, (m, n, k, dt) in enumerate(shapes):
        P, Pr = _make(m, d, k, 1000 * seed + 2 * i)
        Q, Qr = _make(n, d, k, 1000 * seed + 2 * i + 1)
        G = synth.normal((m, n), 1e-3, 5000 * seed + i, dtype=dt).to(DEV)
        g_dtype = native.SF_FP32 if dt == torch.float32 else native.SF_BF16
        S = torch.full((d, d), float("nan"), device=DEV)
        nb = native.lsp_workspace_bytes(m, n, d)
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=DEV)
        native.lsp_compress(P, Q, G, g_dtype, m, n, S, ws, nb)
        torch.cuda.synchronize()
        S_ref, S_abs = ol.compress(Pr, Qr, f64(G.float()))
        check_close(f"S (m={m}, n={n}, k={k}, {dt})", S, S_ref, S_abs, TOL_LSP)
        # decompress-apply into an fp32 W of zeros gives -P dS Q^T
        dS = synth.normal((d, d), 1e-4, 7000 * seed + i).to(DEV)
        W = torch.zeros(m, n, device=DEV)
        native.lsp_decompress_apply(P, Q, dS, W, native.SF_FP32, None, m, n, ws, nb)
        torch.cuda.synchronize()
        D, D_abs = ol.decompress(Pr, Qr, f64(dS))
        check_close(f"-D (m={m}, n={n}, k={k})", W, -D, D_abs, TOL_LSP)
        mats.append((m, n, P, Q, G, g_dtype))
        per.append(S)
    # the same matrices as one layer call: the per-matrix bits
    Ss = [torch.full((d, d), float("nan"), device=DEV) for _ in mats]
    ms, ns = [x[0] for x in mats], [x[1] for x in mats]
    nb = native.lsp_compress_layer_workspace_bytes(ms, ns, d)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    native.lsp_compress_layer([x[2] for x in mats], [x[3] for x in mats], [x[4] for x in mats],
                              [x[5] for x in mats], ms, ns, Ss, ws, nb)
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(Ss, per)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"matrix {i} {shapes[i]}: layer != per-matrix"
    native.sf_sync_status()

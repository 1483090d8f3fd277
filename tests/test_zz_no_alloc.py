"""lsp_compress_noalloc: compress without a caller workspace (GPU).

Some callers cannot allocate device memory or hand over a workspace (a
framework's caching allocator owns the pool, or cudaMalloc's implicit
synchronisation is not acceptable in their loop).  The no-alloc entry point
keeps the compress intermediate in a fixed array inside the library.  These
tests call it through the C ABI on two calls in a row, so the second call
must not be affected by what the first left in the shared array: its S must
be bitwise the S of lsp_compress (which takes a caller workspace), and both
must match the fp64 oracle (oracle/lsp.py) within the projector tolerance,
against the magnitude |P|^T |G| |Q| of S's terms.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from _util import TOL_LSP, check_close, f64
from layer_optimizer_gb300 import native, synth
from oracle import lsp as ol

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _proj(rows, d, k, seed):
    idx, val = synth.projector(rows, d, k, seed)
    return native.lsp_projector_create(rows, d, k, torch.from_numpy(idx).to(DEV), torch.from_numpy(val).to(DEV))


def _reference(P, Q, G, dt, m, n, d):
    S = torch.empty(d, d, device=DEV)
    nb = native.lsp_workspace_bytes(m, n, d)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    native.lsp_compress(P, Q, G, dt, m, n, S, ws, nb)
    torch.cuda.synchronize()
    return S


@pytest.mark.parametrize("m,n,d,k,torch_dt,dt", [
    (4096, 4096, 512, 8, torch.float32, native.SF_FP32),    # LLaMA-7B q-shaped gradient
    (1024, 1024, 64, 4, torch.bfloat16, native.SF_BF16),    # one 1024 x 1024 linear layer, bf16 grads
    (333, 264, 200, 3, torch.float32, native.SF_FP32),      # ragged tiles and outputs (d not a multiple of 4)
])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(m, n, d, k, torch_dt, dt):
    lib = native.load()
    (Pi, Pv), (Qi, Qv) = synth.projector(m, d, k, 1000 + m), synth.projector(n, d, k, 2000 + n)
    P = native.lsp_projector_create(m, d, k, torch.from_numpy(Pi).to(DEV), torch.from_numpy(Pv).to(DEV))
    Q = native.lsp_projector_create(n, d, k, torch.from_numpy(Qi).to(DEV), torch.from_numpy(Qv).to(DEV))
    Po, Qo = ol.Projector(Pi, Pv, d), ol.Projector(Qi, Qv, d)
    for call in range(2):
        G = synth.normal((m, n), 1e-3, 3000 + call, dtype=torch_dt)
        Gd = G.to(DEV)
        S = torch.full((d, d), float("nan"), device=DEV)
        st = lib.lsp_compress_noalloc(P.handle, Q.handle, Gd.data_ptr(), dt, m, n, S.data_ptr(), None)
        assert st == native.SF_OK, native.sf_last_error()
        torch.cuda.synchronize()
        ref = _reference(P, Q, Gd, dt, m, n, d)
        assert torch.equal(S.view(torch.int32), ref.view(torch.int32)), f"call {call + 1}: not the bits of lsp_compress"
        S_ref, S_abs = ol.compress(Po, Qo, f64(G.float()))
        check_close(f"S vs oracle (call {call + 1})", S, S_ref, S_abs, TOL_LSP)
    native.sf_sync_status()


def test_noalloc_rejects_shapes_beyond_the_fixed_scratch():
    lib = native.load()
    m, n, d = 64, 20000, 512          # the intermediate alone is 20000 x 512 fp32 = 41 MB
    assert native.lsp_workspace_bytes(m, n, d) > native.SF_NOALLOC_SCRATCH_BYTES
    P, Q = _proj(m, d, 8, 1), _proj(n, d, 8, 2)
    G = torch.empty(1, device=DEV)    # never read: the size check comes first
    S = torch.empty(d, d, device=DEV)
    st = lib.lsp_compress_noalloc(P.handle, Q.handle, G.data_ptr(), native.SF_FP32, m, n, S.data_ptr(), None)
    assert st == native.SF_ERR_UNSUPPORTED
    assert "scratch" in native.sf_last_error()
    native.sf_sync_status()

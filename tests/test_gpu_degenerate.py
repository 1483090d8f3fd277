"""Degenerate calls: empty tensor lists, zero-element arrays, empty visit orders (GPU).

Each entry point takes its empty case as a no-op: it returns SF_OK, launches
nothing that writes, and leaves the caller's buffers (filled here with guard
values) as they were.
"""

import ctypes

import pytest
import torch

from layer_optimizer_gb300 import native

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _guarded(n, value, dtype=torch.float32, pinned=False):
    t = torch.full((n,), value, dtype=dtype)
    return t.pin_memory() if pinned else t.to(DEV)


def test_adamw_empty_list_and_zero_element_tensors():
    hp = native.hparams()
    native.sf_adamw_layer_step([], hp, 1)
    g = _guarded(8, 7.0, torch.bfloat16)
    p, m, v = _guarded(8, 3.0), _guarded(8, 5.0), _guarded(8, 6.0)
    w = _guarded(8, 9.0, torch.bfloat16)
    native.sf_adamw_layer_step([native.make_tensor(g, p, m, v, w, numel=0)] * 3, hp, 1)
    torch.cuda.synchronize()
    for t, val in ((g, 7.0), (p, 3.0), (m, 5.0), (v, 6.0), (w, 9.0)):
        assert torch.all(t.float() == val)
    native.sf_sync_status()


def test_compressed_adamw_zero_elements():
    S, m, v, dS = _guarded(16, 1.0), _guarded(16, 2.0), _guarded(16, 3.0), _guarded(16, 4.0)
    native.lsp_adamw_compressed(S, m, v, dS, 0, native.hparams(), 1)
    torch.cuda.synchronize()
    for t, val in ((S, 1.0), (m, 2.0), (v, 3.0), (dS, 4.0)):
        assert torch.all(t == val)
    native.sf_sync_status()


def test_layer_window_empty_visit_order():
    n = 64
    slots = [[[_guarded(n, 0.0, torch.bfloat16), _guarded(n, 0.0), _guarded(n, 0.0), _guarded(n, 0.0),
               _guarded(n, 0.0, torch.bfloat16)]] for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.sf_window_create([[native.make_tensor(*t) for t in s] for s in slots], *streams)
    host = [[_guarded(n, 1.0, torch.bfloat16, True), _guarded(n, 2.0, pinned=True), _guarded(n, 3.0, pinned=True),
             _guarded(n, 4.0, pinned=True), _guarded(n, 5.0, torch.bfloat16, True)]]
    layers = native.host_layers([[native.make_tensor(*t) for t in host]])
    steps = (ctypes.c_int64 * 1)(0)
    native.sf_slide_window_step(win, layers, [], native.hparams(), steps)
    torch.cuda.synchronize()
    assert steps[0] == 0
    for t, val in zip(host[0], (1.0, 2.0, 3.0, 4.0, 5.0)):
        assert torch.all(t.float() == val)
    win.close()
    native.sf_sync_status()


@pytest.mark.parametrize("host_update", [False, True])
def test_projector_windows_empty_visit_order(host_update):
    d = 16
    wsb = native.lsp_workspace_bytes(64, 64, d)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=DEV)
    streams = [torch.cuda.Stream() for _ in range(3)]
    S, dS = _guarded(d * d, 1.0), _guarded(d * d, 2.0)
    if host_update:
        Sh, dSh = _guarded(d * d, 3.0, pinned=True), _guarded(d * d, 4.0, pinned=True)
        win = native.lsp_window_create_host_update([(S, dS, Sh, dSh, ws, wsb)], d, *streams)
        bufs = ((S, 1.0), (dS, 2.0), (Sh, 3.0), (dSh, 4.0))
    else:
        m, v = _guarded(d * d, 3.0), _guarded(d * d, 4.0)
        win = native.lsp_window_create([(S, m, v, dS, ws, wsb)], d, *streams)
        bufs = ((S, 1.0), (dS, 2.0), (m, 3.0), (v, 4.0))
    steps = (ctypes.c_int64 * 1)(0)
    native.lsp_slide_window_step(win, native.lsp_layers([]), [], native.hparams(), steps)
    win.sync()
    assert steps[0] == 0
    for t, val in bufs:
        assert torch.all(t == val)
    win.close()
    native.sf_sync_status()

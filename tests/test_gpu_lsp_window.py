"""Sparse-projector step with the compressed moments in pinned host memory (GPU).

The layer-wise engine must give bitwise the results of the same calls with
device-resident moments, whatever the visit order and slot count.
"""

import ctypes

import numpy as np
import pytest
import torch

from _util import HP, TOL_STATE, check_close, f64
from layer_optimizer_gb300 import native, synth
from oracle import adamw as oa

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _proj(rows, d, k, seed):
    idx, val = synth.projector(rows, d, k, seed)
    return native.lsp_projector_create(rows, d, k, torch.from_numpy(idx).to(DEV), torch.from_numpy(val).to(DEV))


def _layers(shapes, d, k, seed, w_bf16):
    out = []
    for i, (m, n, gdt) in enumerate(shapes):
        G = synth.normal((m, n), 1e-3, synth.sub_seed(seed, i, 0), dtype=gdt).to(DEV)
        W0 = synth.normal((m, n), 0.02, synth.sub_seed(seed, i, 1))
        out.append(dict(P=_proj(m, d, k, synth.sub_seed(seed, i, 2)), Q=_proj(n, d, k, synth.sub_seed(seed, i, 3)),
                        G=G, g_dtype=native.SF_FP32 if gdt == torch.float32 else native.SF_BF16,
                        W=(W0.to(torch.bfloat16) if w_bf16 else W0).to(DEV),
                        w_dtype=native.SF_BF16 if w_bf16 else native.SF_FP32, m=m, n=n))
    return out


def _slots(n_slots, d, wsb):
    return [tuple(torch.zeros(d, d, device=DEV) for _ in range(4)) +
            (torch.empty(wsb, dtype=torch.uint8, device=DEV), wsb) for _ in range(n_slots)]


def _resident(layers, order, d, hp):
    """The same sequence of calls with device-resident moments."""
    W = [L["W"].clone() for L in layers]
    mom = [(torch.zeros(d, d, device=DEV), torch.zeros(d, d, device=DEV)) for _ in layers]
    S, dS = torch.empty(d, d, device=DEV), torch.empty(d, d, device=DEV)
    steps = [0] * len(layers)
    for l in order:
        L = layers[l]
        wsb = native.lsp_workspace_bytes(L["m"], L["n"], d)
        ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
        steps[l] += 1
        native.lsp_compress(L["P"], L["Q"], L["G"], L["g_dtype"], L["m"], L["n"], S, ws, wsb)
        native.lsp_adamw_compressed(S, mom[l][0], mom[l][1], dS, d * d, hp, steps[l])
        native.lsp_decompress_apply(L["P"], L["Q"], dS, W[l], L["w_dtype"], None, L["m"], L["n"], ws, wsb)
    torch.cuda.synchronize()
    return W, mom, steps


@pytest.mark.parametrize("n_slots,d,k,w_bf16", [(2, 64, 4, False), (3, 512, 8, True), (1, 96, 3, False)])
def test_lsp_window_matches_resident_bitwise(n_slots, d, k, w_bf16):
    shapes = [(256, 192, torch.float32), (130, 264, torch.bfloat16), (400, 128, torch.float32)]
    layers = _layers(shapes, d, k, 5 + d, w_bf16)
    order = [0, 1, 2, 2, 0, 1, 0]
    hp = native.hparams(**HP)
    W_ref, mom_ref, steps_ref = _resident(layers, order, d, hp)

    for L in layers:
        L["m_host"] = torch.zeros(d, d).pin_memory()
        L["v_host"] = torch.zeros(d, d).pin_memory()
    wsb = max(native.lsp_workspace_bytes(L["m"], L["n"], d) for L in layers)
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.lsp_window_create(_slots(n_slots, d, wsb), d, *streams)
    steps = (ctypes.c_int64 * len(layers))()
    native.lsp_slide_window_step(win, native.lsp_layers(layers), order, hp, steps)
    win.sync()
    assert list(steps) == steps_ref
    for L, Wr, (mr, vr) in zip(layers, W_ref, mom_ref):
        a = L["W"].view(torch.int16 if w_bf16 else torch.int32)
        b = Wr.view(torch.int16 if w_bf16 else torch.int32)
        assert torch.equal(a, b)
        assert torch.equal(L["m_host"].view(torch.int32), mr.cpu().view(torch.int32))
        assert torch.equal(L["v_host"].view(torch.int32), vr.cpu().view(torch.int32))
    win.close()


def test_lsp_window_moments_match_oracle_first_visit():
    d, k = 64, 4
    layers = _layers([(300, 200, torch.float32)], d, k, 99, False)
    L = layers[0]
    L["m_host"] = torch.zeros(d, d).pin_memory()
    L["v_host"] = torch.zeros(d, d).pin_memory()
    wsb = native.lsp_workspace_bytes(L["m"], L["n"], d)
    S_ref = torch.empty(d, d, device=DEV)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    native.lsp_compress(L["P"], L["Q"], L["G"], native.SF_FP32, L["m"], L["n"], S_ref, ws, wsb)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.lsp_window_create(_slots(2, d, wsb), d, *streams)
    steps = (ctypes.c_int64 * 1)()
    native.lsp_slide_window_step(win, native.lsp_layers(layers), [0], native.hparams(**HP), steps)
    win.sync()
    _, m_ref, v_ref, _, m_abs = oa.compressed_adamw_step(f64(S_ref), np.zeros((d, d)), np.zeros((d, d)), 1,
                                                         HP["lr"], HP["beta1"], HP["beta2"], HP["eps"])
    check_close("m~", L["m_host"], m_ref, m_abs, TOL_STATE)
    check_close("v~", L["v_host"], v_ref, v_ref, TOL_STATE)
    win.close()


def test_lsp_window_rejects_bad_layers():
    d = 64
    layers = _layers([(128, 128, torch.float32)], d, 4, 7, False)
    L = layers[0]
    L["m_host"] = torch.zeros(d, d).pin_memory()
    L["v_host"] = torch.zeros(d, d).pin_memory()
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.lsp_window_create(_slots(1, d, 256), d, *streams)     # workspace far too small
    steps = (ctypes.c_int64 * 1)()
    with pytest.raises(native.SfError, match="workspace"):
        native.lsp_slide_window_step(win, native.lsp_layers(layers), [0], native.hparams(**HP), steps)
    with pytest.raises(native.SfError, match="out of"):
        native.lsp_slide_window_step(win, native.lsp_layers(layers), [3], native.hparams(**HP), steps)
    assert steps[0] == 0
    win.close()


def _host_slots(n_slots, d, wsb):
    # device S, dS, workspace; pinned host staging for S and dS
    return [(torch.zeros(d, d, device=DEV), torch.zeros(d, d, device=DEV), torch.zeros(d, d).pin_memory(),
             torch.zeros(d, d).pin_memory(), torch.empty(wsb, dtype=torch.uint8, device=DEV), wsb)
            for _ in range(n_slots)]


@pytest.mark.parametrize("n_slots,d,k,w_bf16,threads", [(2, 64, 4, False, 3), (3, 512, 8, True, 0),
                                                          (1, 96, 3, False, 1), (4, 64, 4, True, 8)])
def test_lsp_host_update_window_matches_resident_bitwise(n_slots, d, k, w_bf16, threads):
    # LSP-Offload's placement: S to the host, the compressed AdamW on host
    # cores, dS back; the same bits as the device-resident chain
    shapes = [(256, 192, torch.float32), (130, 264, torch.bfloat16), (400, 128, torch.float32)]
    layers = _layers(shapes, d, k, 50 + d, w_bf16)
    order = [0, 1, 2, 2, 0, 1, 0, 2, 2, 2]
    hp = native.hparams(**HP)
    W_ref, mom_ref, steps_ref = _resident(layers, order, d, hp)

    for L in layers:
        L["m_host"] = torch.zeros(d, d).pin_memory()
        L["v_host"] = torch.zeros(d, d).pin_memory()
    wsb = max(native.lsp_workspace_bytes(L["m"], L["n"], d) for L in layers)
    streams = [torch.cuda.Stream() for _ in range(3)]
    slots = _host_slots(n_slots, d, wsb)
    win = native.lsp_window_create_host_update(slots, d, *streams, n_threads=threads)
    steps = (ctypes.c_int64 * len(layers))()
    lay = native.lsp_layers(layers)
    native.lsp_slide_window_step(win, lay, order[:4], hp, steps)       # two calls in a row
    native.lsp_slide_window_step(win, lay, order[4:], hp, steps)
    win.sync()
    assert list(steps) == steps_ref
    for L, Wr, (mr, vr) in zip(layers, W_ref, mom_ref):
        a = L["W"].view(torch.int16 if w_bf16 else torch.int32)
        b = Wr.view(torch.int16 if w_bf16 else torch.int32)
        assert torch.equal(a, b)
        assert torch.equal(L["m_host"].view(torch.int32), mr.cpu().view(torch.int32))
        assert torch.equal(L["v_host"].view(torch.int32), vr.cpu().view(torch.int32))
    win.close()
    native.sf_sync_status()


def test_lsp_host_update_window_first_visit_vs_oracle_and_bad_slots():
    d, k = 64, 4
    layers = _layers([(300, 200, torch.float32)], d, k, 98, False)
    L = layers[0]
    L["m_host"] = torch.zeros(d, d).pin_memory()
    L["v_host"] = torch.zeros(d, d).pin_memory()
    wsb = native.lsp_workspace_bytes(L["m"], L["n"], d)
    S_ref = torch.empty(d, d, device=DEV)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    native.lsp_compress(L["P"], L["Q"], L["G"], native.SF_FP32, L["m"], L["n"], S_ref, ws, wsb)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(3)]
    slots = _host_slots(2, d, wsb)
    win = native.lsp_window_create_host_update(slots, d, *streams)
    steps = (ctypes.c_int64 * 1)()
    native.lsp_slide_window_step(win, native.lsp_layers(layers), [0], native.hparams(**HP), steps)
    win.sync()
    dS_ref, m_ref, v_ref, dS_abs, m_abs = oa.compressed_adamw_step(f64(S_ref), np.zeros((d, d)), np.zeros((d, d)),
                                                                  1, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"])
    check_close("m~", L["m_host"], m_ref, m_abs, TOL_STATE)
    check_close("v~", L["v_host"], v_ref, v_ref, TOL_STATE)
    win.close()
    bad = _host_slots(1, d, wsb)
    bad[0] = (bad[0][0], bad[0][1], None, bad[0][3], bad[0][4], bad[0][5])
    with pytest.raises(native.SfError, match="NULL buffer"):
        native.lsp_window_create_host_update(bad, d, *streams)


def test_lsp_host_update_window_timeline_is_causal():
    d, k = 64, 4
    shapes = [(256, 192, torch.float32), (130, 264, torch.float32), (400, 128, torch.float32)]
    layers = _layers(shapes, d, k, 77, False)
    for L in layers:
        L["m_host"] = torch.zeros(d, d).pin_memory()
        L["v_host"] = torch.zeros(d, d).pin_memory()
    wsb = max(native.lsp_workspace_bytes(L["m"], L["n"], d) for L in layers)
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.lsp_window_create_host_update(_host_slots(3, d, wsb), d, *streams)
    native.lsp_window_timeline_start(win, 5)
    steps = (ctypes.c_int64 * 3)()
    native.lsp_slide_window_step(win, native.lsp_layers(layers), [0, 1, 2, 0, 1, 2], native.hparams(**HP), steps)
    win.sync()
    tl = native.lsp_window_timeline_read(win, 16)
    assert len(tl) == 5                                   # capacity 5 of the 6 visits
    for v in tl:
        c0, c1, s0, s1, h1, u0, u1, a0, a1 = v
        assert c0 <= c1 <= s0 <= s1 <= h1 <= u0 <= u1 <= a0 <= a1
    assert tl[0][0] == 0.0
    with pytest.raises(native.SfError, match="host-update"):
        dev = native.lsp_window_create(_slots(1, d, wsb), d, *streams)
        try:
            native.lsp_window_timeline_start(dev, 4)
        finally:
            dev.close()
    win.close()

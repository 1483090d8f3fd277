"""Layer-sliding window engine: results, ordering, failure handling (GPU)."""

import ctypes

import numpy as np
import pytest
import torch

from _util import HP, TOL_STATE, check_close, f64
from layer_optimizer_gb300 import native, synth
from oracle import adamw as oa

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _host_layer(sizes, seed, weight=True):
    out = []
    for i, n in enumerate(sizes):
        g = synth.normal((n,), 1e-3, synth.sub_seed(seed, 0, i), dtype=torch.bfloat16).pin_memory()
        p = synth.normal((n,), 0.02, synth.sub_seed(seed, 1, i)).pin_memory()
        m = torch.zeros(n).pin_memory()
        v = torch.zeros(n).pin_memory()
        w = torch.zeros(n, dtype=torch.bfloat16).pin_memory() if weight else None
        out.append([g, p, m, v, w])
    return out


def _slots(n_slots, caps):
    return [[[torch.empty(c, dtype=torch.bfloat16, device=DEV), torch.empty(c, device=DEV),
              torch.empty(c, device=DEV), torch.empty(c, device=DEV),
              torch.empty(c, dtype=torch.bfloat16, device=DEV)] for c in caps] for _ in range(n_slots)]


def _window(slots, streams):
    sl = [[native.make_tensor(*t) for t in s] for s in slots]
    return native.sf_window_create(sl, *streams)


def _resident_reference(layers, order, grads_per_visit=None):
    """The same visits on device-resident copies with sf_adamw_layer_step."""
    dev = [[[x.to(DEV) if x is not None else None for x in t] for t in L] for L in layers]
    steps = [0] * len(layers)
    hp = native.hparams(**HP)
    for l in order:
        steps[l] += 1
        native.sf_adamw_layer_step([native.make_tensor(*t) for t in dev[l]], hp, steps[l])
    torch.cuda.synchronize()
    return dev, steps


SIZES = [4099, 17, 65536, 3]


def test_window_matches_resident_path_bitwise():
    layers = [_host_layer(SIZES, 10 + l) for l in range(4)]
    ref_in = [[[x.clone() if x is not None else None for x in t] for t in L] for L in layers]
    order = [l % 4 for l in range(12)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = _window(_slots(2, SIZES), streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L] for L in layers])
    steps = (ctypes.c_int64 * 4)()
    native.sf_slide_window_step(win, hl, order, native.hparams(**HP), steps)
    win.sync()
    assert list(steps) == [3, 3, 3, 3]
    ref, ref_steps = _resident_reference(ref_in, order)
    for L, R in zip(layers, ref):
        for t, r in zip(L, R):
            for k in (1, 2, 3):
                assert torch.equal(t[k].view(torch.int32), r[k].cpu().view(torch.int32))
            assert torch.equal(t[4].view(torch.int16), r[4].cpu().view(torch.int16))
    win.close()


def test_window_constant_gradient_closed_form():
    # grads stay fixed in the host slots, so every visit applies the same g
    layers = [_host_layer([20000], 30 + l) for l in range(4)]
    th0 = [f64(L[0][1]) for L in layers]
    g64 = [f64(L[0][0].float()) for L in layers]
    order = [l % 4 for l in range(88)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = _window(_slots(2, [20000]), streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L] for L in layers])
    steps = (ctypes.c_int64 * 4)()
    native.sf_slide_window_step(win, hl, order, native.hparams(**HP), steps)
    win.sync()
    assert list(steps) == [22] * 4
    lam = HP["lr"] * HP["weight_decay"]
    geo = -np.expm1(22 * np.log1p(-lam)) / lam
    for L, t0, g in zip(layers, th0, g64):
        s = g / (np.abs(g) + HP["eps"])
        want = (1 - lam) ** 22 * t0 - HP["lr"] * s * geo
        check_close("theta_22", L[0][1], want, np.abs(t0) + HP["lr"] * geo, TOL_STATE * 22)
    win.close()


def test_window_three_slots_uneven_order_and_no_weight():
    layers = [_host_layer(SIZES[:2], 50 + l, weight=(l % 2 == 0)) for l in range(5)]
    ref_in = [[[x.clone() if x is not None else None for x in t] for t in L] for L in layers]
    order = [0, 2, 2, 4, 1, 0, 3, 3, 3, 1]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = _window(_slots(3, SIZES[:2]), streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L] for L in layers])
    steps = (ctypes.c_int64 * 5)()
    native.sf_slide_window_step(win, hl, order, native.hparams(**HP), steps)
    win.sync()
    ref, ref_steps = _resident_reference(ref_in, order)
    assert list(steps) == ref_steps
    for L, R in zip(layers, ref):
        for t, r in zip(L, R):
            assert torch.equal(t[1].view(torch.int32), r[1].cpu().view(torch.int32))
    win.close()


def test_window_oracle_parity_one_visit():
    layers = [_host_layer([70001, 9], 70)]
    pre = [(f64(t[1]), f64(t[0].float())) for t in layers[0]]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = _window(_slots(2, [70001, 9]), streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in layers[0]]])
    steps = (ctypes.c_int64 * 1)()
    native.sf_slide_window_step(win, hl, [0], native.hparams(**HP), steps)
    win.sync()
    for (th, g), t in zip(pre, layers[0]):
        st = oa.AdamWState(th)
        oa.adamw_step(st, g, 1, **HP)
        check_close("master", t[1], st.theta, st.theta_abs, TOL_STATE)
        check_close("m", t[2], st.m, st.m_abs, TOL_STATE)
    win.close()


def test_injected_copy_failure_leaves_window_usable():
    layers = [_host_layer(SIZES, 90 + l) for l in range(2)]
    ref_in = [[[x.clone() if x is not None else None for x in t] for t in L] for L in layers]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = _window(_slots(2, SIZES), streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L] for L in layers])
    steps = (ctypes.c_int64 * 2)()
    native.sf_test_fail_copy_after(3)   # third h2d copy of the first visit
    with pytest.raises(native.SfError, match="injected"):
        native.sf_slide_window_step(win, hl, [0, 1], native.hparams(**HP), steps)
    assert list(steps) == [0, 0]
    native.sf_test_fail_copy_after(0)
    native.sf_slide_window_step(win, hl, [0, 1], native.hparams(**HP), steps)
    win.sync()
    ref, _ = _resident_reference(ref_in, [0, 1])
    for L, R in zip(layers, ref):
        for t, r in zip(L, R):
            assert torch.equal(t[1].view(torch.int32), r[1].cpu().view(torch.int32))
    win.close()


def test_bounded_wait_times_out_then_recovers():
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = _window(_slots(1, [16]), streams)
    with torch.cuda.stream(streams[1]):
        torch.cuda._sleep(int(3e9))        # a finite spin of ~1.5 s on the compute stream
    with pytest.raises(native.SfError) as e:
        win.sync(timeout_ms=50)
    assert e.value.status == native.SF_ERR_TIMEOUT
    win.sync()                            # default bound: waits for the spin to end
    win.close()


def test_device_wait_runs_out_sets_timeout_and_context_stays_usable():
    # a kernel whose mbarrier wait nothing completes: the bounded wait runs
    # out (~0.1 ms here), records the timeout, and the kernel returns
    native.sf_test_device_wait_runs_out(200_000)
    torch.cuda.synchronize()
    with pytest.raises(native.SfError) as e:
        native.sf_sync_status()
    assert e.value.status == native.SF_ERR_TIMEOUT and "ran out" in str(e.value)
    native.sf_sync_status()                       # the word was cleared
    # the context still works: an AdamW step runs and checks out
    n = 4096
    g = torch.full((n,), 1e-3, dtype=torch.bfloat16, device="cuda")
    p, m, v = torch.ones(n, device="cuda"), torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    native.sf_adamw_layer_step([native.make_tensor(g, p, m, v, None, n)], native.hparams(**HP), 1)
    torch.cuda.synchronize()
    native.sf_sync_status()
    assert torch.all(p < 1.0)
    with pytest.raises(native.SfError, match="limit_cycles"):
        native.sf_test_device_wait_runs_out(0)


def test_invalid_visits_rejected_before_enqueue():
    layers = [_host_layer([100], 99)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = _window(_slots(2, [50]), streams)   # slot too small
    hl = native.host_layers([[native.make_tensor(*t) for t in layers[0]]])
    steps = (ctypes.c_int64 * 1)()
    with pytest.raises(native.SfError, match="capacity"):
        native.sf_slide_window_step(win, hl, [0], native.hparams(**HP), steps)
    with pytest.raises(native.SfError, match="out of"):
        native.sf_slide_window_step(win, hl, [1], native.hparams(**HP), steps)
    assert steps[0] == 0
    win.close()


def _flat_layer(sizes, seed, no_weight=()):
    """A layer kept as one pinned buffer per array, the tensors views into it."""
    tot = sum(sizes)
    flat = [torch.zeros(tot, dtype=dt).pin_memory()
            for dt in (torch.bfloat16, torch.float32, torch.float32, torch.float32, torch.bfloat16)]
    out, o = [], 0
    for i, n in enumerate(sizes):
        t = [f[o:o + n] for f in flat]
        t[0].copy_(synth.normal((n,), 1e-3, synth.sub_seed(seed, 0, i), dtype=torch.bfloat16))
        t[1].copy_(synth.normal((n,), 0.02, synth.sub_seed(seed, 1, i)))
        if i in no_weight:
            t[4] = None
        out.append(t)
        o += n
    return out


def test_window_flat_layers_copy_as_runs_bitwise():
    # contiguous host arrays and contiguous slot arrays move as one copy per
    # run; a missing weight and a slot tensor with spare capacity end runs
    sizes = [4099, 17, 65536, 3, 1024]
    layers = [_flat_layer(sizes, 200 + l, no_weight=(2,) if l == 1 else ()) for l in range(3)]
    ref_in = [[[x.clone() if x is not None else None for x in t] for t in L] for L in layers]
    caps = list(sizes)
    caps[3] = 8                                     # spare capacity: tensors 3 and 4 are not adjacent in the slot
    slots = []
    for _ in range(2):
        flat = [torch.empty(sum(caps), dtype=dt, device=DEV)
                for dt in (torch.bfloat16, torch.float32, torch.float32, torch.float32, torch.bfloat16)]
        sl, o = [], 0
        for c in caps:
            sl.append([f[o:o + c] for f in flat])
            o += c
        slots.append(sl)
    order = [0, 1, 2, 1, 0, 2, 2]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = _window(slots, streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L] for L in layers])
    steps = (ctypes.c_int64 * 3)()
    native.sf_slide_window_step(win, hl, order, native.hparams(**HP), steps)
    win.sync()
    ref, ref_steps = _resident_reference(ref_in, order)
    assert list(steps) == ref_steps
    for L, R in zip(layers, ref):
        for t, r in zip(L, R):
            for k in (1, 2, 3):
                assert torch.equal(t[k].view(torch.int32), r[k].cpu().view(torch.int32))
            if t[4] is not None:
                assert torch.equal(t[4].view(torch.int16), r[4].cpu().view(torch.int16))
    win.close()


def test_window_with_device_resident_states_moves_only_grads_and_weights():
    # fp32 master, m and v live in HBM; gradients come from and bf16 weights go
    # back to pinned host memory; the slots hold only grad and weight buffers
    sizes = [4099, 17, 65536, 3]
    layers = []
    for l in range(3):
        L = _host_layer(sizes, 90 + l)
        layers.append([[t[0], t[1].to(DEV), t[2].to(DEV), t[3].to(DEV), t[4]] for t in L])
    ref_in = [[[x.clone() if x is not None else None for x in t] for t in L] for L in layers]
    torch.cuda.synchronize()          # the clones are taken before the window's streams touch the states
    order = [0, 1, 2, 2, 0, 1, 1]
    bufs = [[(torch.empty(c, dtype=torch.bfloat16, device=DEV), torch.empty(c, dtype=torch.bfloat16, device=DEV))
             for c in sizes] for _ in range(2)]          # kept alive: the window holds raw addresses
    slots = [[native.make_tensor(g, None, None, None, w, numel=g.numel()) for g, w in sb] for sb in bufs]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.sf_window_create(slots, *streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L] for L in layers])
    steps = (ctypes.c_int64 * 3)()
    native.sf_slide_window_step(win, hl, order, native.hparams(**HP), steps)
    win.sync()
    torch.cuda.synchronize()
    ref, ref_steps = _resident_reference(ref_in, order)
    assert list(steps) == ref_steps
    for L, R in zip(layers, ref):
        for t, r in zip(L, R):
            for k in (1, 2, 3):
                assert t[k].is_cuda
                assert torch.equal(t[k].view(torch.int32), r[k].view(torch.int32))
            assert not t[4].is_cuda
            assert torch.equal(t[4].view(torch.int16), r[4].cpu().view(torch.int16))
    win.close()
    del bufs


def test_window_rejects_host_array_without_slot_buffer():
    sizes = [1024]
    L = _host_layer(sizes, 95)                       # master in pinned host memory
    g, w = torch.empty(1024, dtype=torch.bfloat16, device=DEV), torch.empty(1024, dtype=torch.bfloat16, device=DEV)
    slots = [[native.make_tensor(g, None, None, None, w, numel=1024)]]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.sf_window_create(slots, *streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L]])
    steps = (ctypes.c_int64 * 1)()
    with pytest.raises(native.SfError, match="slot has no buffer"):
        native.sf_slide_window_step(win, hl, [0], native.hparams(**HP), steps)
    assert list(steps) == [0]
    win.close()

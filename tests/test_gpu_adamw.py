"""Parity of the fused multi-tensor AdamW kernel with the fp64 oracle (GPU)."""

import numpy as np
import pytest
import torch

from _util import HP, TOL_STATE, bits, check_bf16, check_close, f64
from layer_optimizer_gb300 import native, synth
from oracle import adamw as oa

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _layer(sizes, seed, offset_elems=0):
    """Device buffers for a layer; optional element offset into larger buffers (misalignment)."""
    out = []
    for i, n in enumerate(sizes):
        o = offset_elems
        g = torch.empty(n + o, dtype=torch.bfloat16, device=DEV)[o:]
        p = torch.empty(n + o, device=DEV)[o:]
        p.copy_(synth.normal((n,), 0.02, synth.sub_seed(seed, 0, i)))
        m = torch.zeros(n + o, device=DEV)[o:]
        v = torch.zeros(n + o, device=DEV)[o:]
        w = torch.empty(n + o, dtype=torch.bfloat16, device=DEV)[o:]
        out.append([g, p, m, v, w])
    return out


def _run_and_check(sizes, steps=3, seed=0, offset=0, grads=None, with_weight=True):
    lay = _layer(sizes, seed, offset)
    states = [oa.AdamWState(f64(x[1])) for x in lay]
    hp = native.hparams(**HP)
    for t in range(1, steps + 1):
        for i, n in enumerate(sizes):
            g = grads(i, t) if grads else synth.normal((n,), 1e-3, synth.sub_seed(seed, 1, i, t),
                                                        dtype=torch.bfloat16)
            lay[i][0].copy_(g)
        # one-step parity: the oracle starts from the kernel's own previous state
        pre = [(f64(x[1]), f64(x[2]), f64(x[3])) for x in lay]
        ts = [native.make_tensor(x[0], x[1], x[2], x[3], x[4] if with_weight else None) for x in lay]
        native.sf_adamw_layer_step(ts, hp, t)
        torch.cuda.synchronize()
        for i, x in enumerate(lay):
            st = oa.AdamWState(pre[i][0], pre[i][1], pre[i][2])
            st.m_abs, st.v_abs, st.theta_abs = states[i].m_abs, states[i].v_abs, np.abs(pre[i][0])
            g64 = f64(x[0].float())
            wref = oa.adamw_step(st, g64, t, **HP)
            oa.adamw_step(states[i], g64, t, **HP)
            check_close(f"master[{i}] t={t}", x[1], st.theta, st.theta_abs, TOL_STATE)
            check_close(f"m[{i}] t={t}", x[2], st.m, st.m_abs, TOL_STATE)
            check_close(f"v[{i}] t={t}", x[3], st.v, st.v_abs, TOL_STATE)
            if with_weight:
                check_bf16(f"w[{i}] t={t}", bits(x[4]), st.theta)
    # chained drift over all steps stays within t x the one-step bound
    for i, x in enumerate(lay):
        check_close(f"master[{i}] chained", x[1], states[i].theta, states[i].theta_abs, TOL_STATE * steps)
    return lay


def test_one_linear_layer_1024x1024_three_steps():
    _run_and_check([1024 * 1024], steps=3)


def test_ragged_sizes_and_many_tensors():
    sizes = [1, 2, 7, 8, 9, 15, 16, 17, 255, 4095, 4096, 4097, 8191, 100003, 0, 3]
    _run_and_check(sizes, steps=2, seed=1)


def test_more_tensors_than_one_launch_holds():
    sizes = [37 + 13 * i for i in range(native.SF_MAX_TENSORS_PER_LAUNCH + 9)]
    _run_and_check(sizes, steps=2, seed=2)


@pytest.mark.parametrize("offset", [1, 3, 4, 5])
def test_misaligned_pointers(offset):
    # all arrays shifted by the same element count: bf16 and fp32 offsets
    # differ in bytes, so some offsets keep a common 16-byte phase and some don't
    _run_and_check([5000, 33, 70001], steps=2, seed=3, offset=offset)


@pytest.mark.parametrize("offset", [0, 3, 4])
def test_bulk_copy_path_with_heads_tails_and_scalar_tensors(offset):
    # over 2^20 aligned elements in one launch: the aligned middles go through
    # the bulk-copy kernel, heads / tails and odd-phase tensors through the
    # register-staged one
    _run_and_check([600001, 500007, 33, 9, 2048 * 3], steps=2, seed=11, offset=offset)


def test_bulk_copy_path_without_weights():
    _run_and_check([1 << 20, 4096 + 3], steps=2, seed=12, with_weight=False)


def test_no_weight_output():
    _run_and_check([3000, 12345], steps=2, seed=4, with_weight=False)


def test_constant_gradient_closed_form_22_steps():
    n = 50000
    g = synth.normal((n,), 1e-3, 77, dtype=torch.bfloat16).to(DEV)
    lay = _layer([n], 5)
    th0 = f64(lay[0][1])
    hp = native.hparams(**HP)
    for t in range(1, 23):
        lay[0][0].copy_(g)
        native.sf_adamw_layer_step([native.make_tensor(*lay[0])], hp, t)
    torch.cuda.synchronize()
    lam = HP["lr"] * HP["weight_decay"]
    g64 = f64(g.float())
    s = g64 / (np.abs(g64) + HP["eps"])
    geo = -np.expm1(22 * np.log1p(-lam)) / lam
    want = (1 - lam) ** 22 * th0 - HP["lr"] * s * geo
    mag = np.abs(th0) + HP["lr"] * geo
    check_close("closed form t=22", lay[0][1], want, mag, TOL_STATE * 22)


def test_special_values():
    n = 64
    lay = _layer([n], 6)
    g = torch.zeros(n, dtype=torch.bfloat16)
    g[1] = float("inf")
    g[2] = float("nan")
    g[3] = -1e30
    g[4] = 1e-40  # bf16 subnormal
    lay[0][0].copy_(g)
    native.sf_adamw_layer_step([native.make_tensor(*lay[0])], native.hparams(**HP), 1)
    torch.cuda.synchronize()
    p = lay[0][1].cpu()
    assert torch.isnan(p[1]) and torch.isnan(p[2])       # inf/inf -> nan propagates, no skipping
    assert torch.isfinite(p[0]) and torch.isfinite(p[3]) and torch.isfinite(p[4])


def test_deterministic_repeat():
    a = _run_and_check([123457], steps=1, seed=8)
    b = _run_and_check([123457], steps=1, seed=8)
    for x, y in zip(a[0], b[0]):
        assert torch.equal(x.view(torch.uint8) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.uint8) if y.dtype == torch.bfloat16 else y.view(torch.int32))


def test_guard_bands_untouched():
    # 4 KiB canaries before and after every array
    n, pad = 10007, 1024
    bufs = [torch.full((n + 2 * pad,), 12345.0, device=DEV) for _ in range(3)]
    gb = torch.full((n + 2 * pad,), 3.0, dtype=torch.bfloat16, device=DEV)
    wb = torch.full((n + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    t = native.make_tensor(gb[pad:pad + n], bufs[0][pad:pad + n], bufs[1][pad:pad + n], bufs[2][pad:pad + n],
                           wb[pad:pad + n])
    native.sf_adamw_layer_step([t], native.hparams(**HP), 1)
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.all(b[:pad] == 12345.0) and torch.all(b[pad + n:] == 12345.0)
    assert torch.all(wb[:pad] == 7.0) and torch.all(wb[pad + n:] == 7.0)
    assert torch.all(gb == 3.0)


def test_invalid_arguments_raise():
    lay = _layer([10], 9)
    t = native.make_tensor(*lay[0])
    with pytest.raises(native.SfError):
        native.sf_adamw_layer_step([t], native.hparams(**HP), 0)
    bad = native.make_tensor(None, lay[0][1], lay[0][2], lay[0][3], None)
    with pytest.raises(native.SfError):
        native.sf_adamw_layer_step([bad], native.hparams(**HP), 1)


@pytest.mark.slow
def test_opt13_stack_sampled():
    """All 24 OPT-1.3B layers, one fused step per layer, checked on sampled elements."""
    layer = synth.OPT13_LAYER
    hp = native.hparams(**HP)
    rng = np.random.default_rng(0)
    for li in range(synth.OPT13_LAYERS):
        bufs = []
        for ti, (_, n) in enumerate(layer):
            g = synth.fill_normal_(torch.empty(n, dtype=torch.bfloat16, device=DEV), 1e-3, synth.sub_seed(1, li, ti))
            p = synth.fill_normal_(torch.empty(n, device=DEV), 0.02, synth.sub_seed(2, li, ti))
            bufs.append([g, p, torch.zeros(n, device=DEV), torch.zeros(n, device=DEV),
                         torch.empty(n, dtype=torch.bfloat16, device=DEV)])
        idx = [torch.from_numpy(np.unique(np.concatenate([
            rng.integers(0, n, 20000), np.arange(min(n, 4096)), np.arange(max(0, n - 4096), n)]))).to(DEV)
            for _, n in layer]
        pre = [(f64(b[1][ix]), f64(b[0][ix].float())) for b, ix in zip(bufs, idx)]
        native.sf_adamw_layer_step([native.make_tensor(*b) for b in bufs], hp, 1)
        torch.cuda.synchronize()
        for (th, g64), b, ix in zip(pre, bufs, idx):
            st = oa.AdamWState(th)
            wref = oa.adamw_step(st, g64, 1, **HP)
            check_close("master", b[1][ix], st.theta, st.theta_abs, TOL_STATE)
            check_close("m", b[2][ix], st.m, st.m_abs, TOL_STATE)
            check_close("v", b[3][ix], st.v, st.v_abs, TOL_STATE)
            check_bf16("w", bits(b[4][ix]), st.theta)
        del bufs


@pytest.mark.slow
def test_tensor_beyond_2_31_elements_sampled():
    """One tensor of 2^31 + 4099 elements (34 GB of arrays), offset by 3 elements so it has a scalar head
    and tail around the bulk-copied middle; checked on sampled elements, across the 2^31 boundary."""
    n, o = 2 ** 31 + 4099, 3
    g = synth.fill_normal_(torch.empty(n + o, dtype=torch.bfloat16, device=DEV), 1e-3, synth.sub_seed(41, 0))[o:]
    p = synth.fill_normal_(torch.empty(n + o, device=DEV), 0.02, synth.sub_seed(41, 1))[o:]
    m = torch.zeros(n + o, device=DEV)[o:]
    v = torch.zeros(n + o, device=DEV)[o:]
    w = torch.empty(n + o, dtype=torch.bfloat16, device=DEV)[o:]
    rng = np.random.default_rng(41)
    ix = torch.from_numpy(np.unique(np.concatenate([
        rng.integers(0, n, 1 << 16), np.arange(64), np.arange(n - 4096, n),
        np.arange(2 ** 31 - 64, 2 ** 31 + 64)]))).to(DEV)
    th, g64 = f64(p[ix]), f64(g[ix].float())
    native.sf_adamw_layer_step([native.make_tensor(g, p, m, v, w)], native.hparams(**HP), 1)
    torch.cuda.synchronize()
    st = oa.AdamWState(th)
    oa.adamw_step(st, g64, 1, **HP)
    check_close("master", p[ix], st.theta, st.theta_abs, TOL_STATE)
    check_close("m", m[ix], st.m, st.m_abs, TOL_STATE)
    check_close("v", v[ix], st.v, st.v_abs, TOL_STATE)
    check_bf16("w", bits(w[ix]), st.theta)
    del g, p, m, v, w
    torch.cuda.empty_cache()
    native.sf_sync_status()


def test_checkpoint_resume_bitwise():
    """Three steps uninterrupted equal: one step, save to host, reload into new buffers, two steps."""
    n = 200003
    grads = [synth.normal((n,), 1e-3, synth.sub_seed(21, t), dtype=torch.bfloat16) for t in (1, 2, 3)]
    hp = native.hparams(**HP)

    def fresh(theta, m=None, v=None):
        return [torch.empty(n, dtype=torch.bfloat16, device=DEV), theta.to(DEV).clone(),
                (torch.zeros(n) if m is None else m).to(DEV).clone(),
                (torch.zeros(n) if v is None else v).to(DEV).clone(),
                torch.empty(n, dtype=torch.bfloat16, device=DEV)]

    theta0 = synth.normal((n,), 0.02, 22)
    a = fresh(theta0)
    for t in (1, 2, 3):
        a[0].copy_(grads[t - 1])
        native.sf_adamw_layer_step([native.make_tensor(*a)], hp, t)
    b = fresh(theta0)
    b[0].copy_(grads[0])
    native.sf_adamw_layer_step([native.make_tensor(*b)], hp, 1)
    saved = [x.cpu().clone() for x in b[1:4]]            # the caller-owned state: master, m, v (and t = 1)
    del b
    c = fresh(*saved)
    for t in (2, 3):
        c[0].copy_(grads[t - 1])
        native.sf_adamw_layer_step([native.make_tensor(*c)], hp, t)
    torch.cuda.synchronize()
    for x, y in zip(a[1:4], c[1:4]):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(a[4].view(torch.int16), c[4].view(torch.int16))


def test_host_step_bitwise_equals_device_step():
    """The host-core update and the device kernels give the same bits (finite inputs)."""
    sizes = [1 << 20, 4097, 33, 600001]
    dev = _layer(sizes, 31)
    host = [[x.cpu().clone() for x in t] for t in dev]
    hp = native.hparams(**HP)
    for t in (1, 2):
        for i, n in enumerate(sizes):
            g = synth.normal((n,), 1e-3, synth.sub_seed(31, 9, i, t), dtype=torch.bfloat16)
            dev[i][0].copy_(g)
            host[i][0].copy_(g)
        native.sf_adamw_layer_step([native.make_tensor(*x) for x in dev], hp, t)
        native.sf_adamw_host_step([native.make_tensor(*x) for x in host], hp, t)
    torch.cuda.synchronize()
    for d_, h_ in zip(dev, host):
        for k in (1, 2, 3):
            assert torch.equal(d_[k].cpu().view(torch.int32), h_[k].view(torch.int32))
        assert torch.equal(d_[4].cpu().view(torch.int16), h_[4].view(torch.int16))


def test_pinned_host_arrays_updated_in_place_bitwise_equal_to_device():
    # arrays in pinned host memory are updated over the host link by the
    # same arithmetic (zero-copy loads and stores); large enough that device
    # arrays of the same sizes take the bulk-copy kernel
    sizes = [(1 << 20) + 8, 3000, 1 << 19]
    hp = native.hparams(**HP)
    dev, host = [], []
    for i, n in enumerate(sizes):
        g = synth.normal((n,), 1e-3, synth.sub_seed(40, i), dtype=torch.bfloat16)
        p = synth.normal((n,), 0.02, synth.sub_seed(41, i))
        dev.append([g.cuda(), p.cuda(), torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda"),
                    torch.empty(n, dtype=torch.bfloat16, device="cuda")])
        host.append([g.pin_memory(), p.pin_memory(), torch.zeros(n).pin_memory(), torch.zeros(n).pin_memory(),
                     torch.empty(n, dtype=torch.bfloat16).pin_memory()])
    for step in (1, 2):
        native.sf_adamw_layer_step([native.make_tensor(*t) for t in dev], hp, step)
        native.sf_adamw_layer_step([native.make_tensor(*t) for t in host], hp, step)
    torch.cuda.synchronize()
    native.sf_sync_status()
    for d, h in zip(dev, host):
        for a, b in zip(d[1:4], h[1:4]):
            assert torch.equal(a.cpu().view(torch.int32), b.view(torch.int32))
        assert torch.equal(d[4].cpu().view(torch.int16), h[4].view(torch.int16))

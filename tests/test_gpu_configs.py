"""Full-size workloads, checked on sampled elements against the fp64 oracle (GPU, slow).

AdamW is elementwise, so checking a sample of elements is exact for those
elements: every tensor contributes ~20k random indices plus its first and
last 4096 elements.
"""

import ctypes
import os

import numpy as np
import pytest
import torch

from _util import HP, TOL_STATE, bits, check_bf16, check_close, f64
from layer_optimizer_gb300 import native, synth
from oracle import adamw as oa

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"


def _sample_idx(n, rng):
    idx = np.unique(np.concatenate([rng.integers(0, n, 20000), np.arange(min(n, 4096)),
                                    np.arange(max(0, n - 4096), n)]))
    return torch.from_numpy(idx)


def _check_step(pre, post, g64, t, what):
    th, m, v = pre
    st = oa.AdamWState(th, m, v)
    oa.adamw_step(st, g64, t, **HP)
    check_close(f"{what} master", post[0], st.theta, st.theta_abs, TOL_STATE)
    check_close(f"{what} m", post[1], st.m, st.m_abs, TOL_STATE)
    check_close(f"{what} v", post[2], st.v, st.v_abs, TOL_STATE)
    check_bf16(f"{what} w", post[3], st.theta)


def test_llama2_7b_full_step_sampled():
    """All 6,738,415,616 params resident; the workload's ten steps in sliding order, fresh gradients each step."""
    groups = synth.llama7_step_order()
    assert sum(synth.layer_numel(g) for g in groups) == 6738415616
    rng = np.random.default_rng(0)
    bufs, idx = [], []
    for li, grp in enumerate(groups):
        ts, ix = [], []
        for ti, (_, n) in enumerate(grp):
            p = synth.fill_normal_(torch.empty(n, device=DEV), 0.02, synth.sub_seed(3, li, ti))
            ts.append([torch.empty(n, dtype=torch.bfloat16, device=DEV), p, torch.zeros(n, device=DEV),
                       torch.zeros(n, device=DEV), torch.empty(n, dtype=torch.bfloat16, device=DEV)])
            ix.append(_sample_idx(n, rng).to(DEV))
        bufs.append(ts)
        idx.append(ix)
    hp = native.hparams(**HP)
    for t in range(1, 11):
        pre = []
        for li, grp in enumerate(groups):
            for ti, (_, n) in enumerate(grp):
                synth.fill_normal_(bufs[li][ti][0], 1e-3, synth.sub_seed(4, li, ti, t))
        for li in range(len(groups)):
            pre.append([(f64(b[1][ix]), f64(b[2][ix]), f64(b[3][ix]), f64(b[0][ix].float()))
                        for b, ix in zip(bufs[li], idx[li])])
        for li in range(len(groups)):
            native.sf_adamw_layer_step([native.make_tensor(*b) for b in bufs[li]], hp, t)
        torch.cuda.synchronize()
        for li in range(len(groups)):
            for ti, (b, ix) in enumerate(zip(bufs[li], idx[li])):
                th, m, v, g64 = pre[li][ti]
                post = (b[1][ix], b[2][ix], b[3][ix], bits(b[4][ix]))
                _check_step((th, m, v), post, g64, t, f"group {li} tensor {ti} t={t}")
    del bufs
    torch.cuda.empty_cache()


def _host_gb():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) / 1e6
    except OSError:
        pass
    return 0.0


@pytest.mark.skipif(_host_gb() < 160, reason="needs ~90 GB of pinned host memory")
def test_mistral_large_window_sampled():
    """Four 1.38 B-param layers in pinned host memory, 2 device slots, the full 88-visit sweep.

    The gradients stay fixed in the host slots, so each layer takes 22
    AdamW steps with the same g; the oracle runs the same 22 steps on the
    sampled elements (chained: the fp32 state may drift from the fp64 one by
    one rounding per step).
    """
    layer = synth.MISTRAL_LAYER
    caps = [n for _, n in layer]
    rng = np.random.default_rng(1)
    host, idx = [], []
    for li in range(4):
        ts, ix = [], []
        for ti, n in enumerate(caps):
            g = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
            g.copy_(synth.fill_normal_(torch.empty(n, dtype=torch.bfloat16, device=DEV), 1e-3,
                                       synth.sub_seed(6, li, ti, 0)))
            p = torch.empty(n, pin_memory=True)
            p.copy_(synth.fill_normal_(torch.empty(n, device=DEV), 0.02, synth.sub_seed(6, li, ti, 1)))
            m = torch.empty(n, pin_memory=True)
            m.copy_(torch.zeros(n, device=DEV))
            v = torch.empty(n, pin_memory=True)
            v.copy_(torch.zeros(n, device=DEV))
            ts.append([g, p, m, v, torch.empty(n, dtype=torch.bfloat16, pin_memory=True)])
            ix.append(_sample_idx(n, rng))
        host.append(ts)
        idx.append(ix)
    slots = [[[torch.empty(c, dtype=torch.bfloat16, device=DEV), torch.empty(c, device=DEV),
               torch.empty(c, device=DEV), torch.empty(c, device=DEV),
               torch.empty(c, dtype=torch.bfloat16, device=DEV)] for c in caps] for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.sf_window_create([[native.make_tensor(*t) for t in s_] for s_ in slots], *streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L] for L in host])
    steps = (ctypes.c_int64 * 4)()
    hp = native.hparams(**HP)
    pre = [[(f64(b[1][ix]), f64(b[2][ix]), f64(b[3][ix]), f64(b[0][ix].float())) for b, ix in zip(L, I)]
           for L, I in zip(host, idx)]
    native.sf_slide_window_step(win, hl, [v % 4 for v in range(88)], hp, steps)
    win.sync()
    assert list(steps) == [22] * 4
    for li in range(4):
        for ti, (b, ix) in enumerate(zip(host[li], idx[li])):
            th, m, v, g64 = pre[li][ti]
            st = oa.AdamWState(th, m, v)
            for t in range(1, 23):
                oa.adamw_step(st, g64, t, **HP)
            what = f"layer {li} tensor {ti} after 22 visits"
            check_close(f"{what} master", b[1][ix], st.theta, st.theta_abs, TOL_STATE * 22)
            check_close(f"{what} m", b[2][ix], st.m, st.m_abs, TOL_STATE * 22)
            check_close(f"{what} v", b[3][ix], st.v, st.v_abs, TOL_STATE * 22)
            # chained: the bf16 weight is the kernel's own fp32 master rounded
            # to nearest even (exactly), the master being within the bound above
            check_bf16(f"{what} w", bits(b[4][ix]), f64(b[1][ix]), max_ulp=0)
    win.close()
    del host, slots
    torch.cuda.empty_cache()
    f = getattr(torch._C, "_host_emptyCache", None)
    if f is not None:
        f()

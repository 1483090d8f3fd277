"""The multi-threaded host AdamW against the fp64 oracle (CPU only: no GPU needed)."""

import numpy as np
import pytest
import torch

from _util import HP, TOL_STATE, bits, check_bf16, check_close, f64
from layer_optimizer_gb300 import build, native, synth
from oracle import adamw as oa


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    native.load()


def _host_layer(sizes, seed):
    out = []
    for i, n in enumerate(sizes):
        out.append([synth.normal((n,), 1e-3, synth.sub_seed(seed, 0, i), dtype=torch.bfloat16),
                    synth.normal((n,), 0.02, synth.sub_seed(seed, 1, i)), torch.zeros(n), torch.zeros(n),
                    torch.empty(n, dtype=torch.bfloat16)])
    return out


@pytest.mark.parametrize("threads", [1, 3, 0])
def test_host_step_matches_oracle(threads):
    sizes = [1, 7, 4097, 100003, 0, 65536 * 3 + 5]
    lay = _host_layer(sizes, 4)
    states = [oa.AdamWState(f64(x[1])) for x in lay]
    hp = native.hparams(**HP)
    for t in (1, 2, 3):
        for i, n in enumerate(sizes):
            lay[i][0].copy_(synth.normal((n,), 1e-3, synth.sub_seed(4, 2, i, t), dtype=torch.bfloat16))
        pre = [(f64(x[1]), f64(x[2]), f64(x[3])) for x in lay]
        native.sf_adamw_host_step([native.make_tensor(*x) for x in lay], hp, t, threads)
        for i, x in enumerate(lay):
            st = oa.AdamWState(*pre[i])
            st.m_abs, st.v_abs = states[i].m_abs, states[i].v_abs
            g64 = f64(x[0].float())
            oa.adamw_step(st, g64, t, **HP)
            oa.adamw_step(states[i], g64, t, **HP)
            check_close(f"master[{i}] t={t}", x[1], st.theta, st.theta_abs, TOL_STATE)
            check_close(f"m[{i}] t={t}", x[2], st.m, st.m_abs, TOL_STATE)
            check_close(f"v[{i}] t={t}", x[3], st.v, st.v_abs, TOL_STATE)
            check_bf16(f"w[{i}] t={t}", bits(x[4]), st.theta)


def test_host_step_thread_count_does_not_change_bits():
    sizes = [300007, 5, 123456]
    a, b = _host_layer(sizes, 5), _host_layer(sizes, 5)
    hp = native.hparams(**HP)
    native.sf_adamw_host_step([native.make_tensor(*x) for x in a], hp, 1, 1)
    native.sf_adamw_host_step([native.make_tensor(*x) for x in b], hp, 1, 7)
    for x, y in zip(a, b):
        for u, w in zip(x[1:], y[1:]):
            assert torch.equal(u.view(torch.int16) if u.dtype == torch.bfloat16 else u.view(torch.int32),
                               w.view(torch.int16) if w.dtype == torch.bfloat16 else w.view(torch.int32))


def test_host_step_rejects_bad_arguments():
    lay = _host_layer([10], 6)
    with pytest.raises(native.SfError):
        native.sf_adamw_host_step([native.make_tensor(*lay[0])], native.hparams(**HP), 0)
    bad = native.make_tensor(None, lay[0][1], lay[0][2], lay[0][3], None)
    with pytest.raises(native.SfError):
        native.sf_adamw_host_step([bad], native.hparams(**HP), 1)


def test_bf16_rounding_of_special_values():
    x = torch.tensor([0.0, -0.0, 1.0, float("inf"), -float("inf"), 3.3895313892515355e38, 1e-40])
    n = x.numel()
    # theta = x exactly after a zero-gradient step with no decay and lr 0
    lay = [[torch.zeros(n, dtype=torch.bfloat16), x.clone(), torch.zeros(n), torch.zeros(n),
            torch.empty(n, dtype=torch.bfloat16)]]
    native.sf_adamw_host_step([native.make_tensor(*lay[0])], native.hparams(lr=0.0, weight_decay=0.0), 1, 1)
    assert torch.equal(lay[0][4].view(torch.int16), x.to(torch.bfloat16).view(torch.int16))

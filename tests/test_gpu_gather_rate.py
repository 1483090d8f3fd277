"""The on-chip gather-rate probes (shared memory and tensor memory: the projector kernels' second roofs) run and reject bad arguments (GPU)."""

import pytest
import torch

from layer_optimizer_gb300 import native

pytestmark = pytest.mark.gpu


def test_gather_rate_probe_runs_and_fills_its_sink():
    sink = torch.full((3 * 512,), float("nan"), device="cuda")
    native.sf_bench_gather_rate(3, 64, sink)
    torch.cuda.synchronize()
    native.sf_sync_status()
    assert bool(torch.isfinite(sink).all()) and bool((sink > 0).all())
    first = sink.clone()
    native.sf_bench_gather_rate(3, 64, sink)
    torch.cuda.synchronize()
    assert torch.equal(first, sink)                   # fixed data: the same sums every time


def test_gather_rate_probe_rejects_bad_arguments():
    sink = torch.empty(512, device="cuda")
    for ctas, iters in ((0, 8), (1, 0)):
        with pytest.raises(native.SfError, match="ctas and iters"):
            native.sf_bench_gather_rate(ctas, iters, sink)


@pytest.mark.parametrize("x", [1, 2, 4])
@pytest.mark.parametrize("entries", [0, 1])
def test_tmem_rate_probe_runs_and_is_repeatable(x, entries):
    sink = torch.full((2 * 512,), float("nan"), device="cuda")
    native.sf_bench_tmem_rate(2, 32, x, entries, sink)
    torch.cuda.synchronize()
    native.sf_sync_status()
    assert bool(torch.isfinite(sink).all()) and bool((sink > 0).all())
    first = sink.clone()
    native.sf_bench_tmem_rate(2, 32, x, entries, sink)
    torch.cuda.synchronize()
    assert torch.equal(first, sink)


def test_tmem_rate_probe_rejects_bad_arguments():
    sink = torch.empty(512, device="cuda")
    with pytest.raises(native.SfError, match="ctas and iters"):
        native.sf_bench_tmem_rate(0, 8, 1, 1, sink)
    with pytest.raises(native.SfError, match="x must be"):
        native.sf_bench_tmem_rate(1, 8, 3, 1, sink)


def test_l2_gather_rate_probe_runs_and_rejects_bad_arguments():
    buf = torch.rand(4096, 128, device="cuda")
    sink = torch.full((3 * 256,), float("nan"), device="cuda")
    native.sf_bench_l2_gather_rate(3, 8, buf, 4096, sink)
    torch.cuda.synchronize()
    native.sf_sync_status()
    assert bool(torch.isfinite(sink).all())
    with pytest.raises(native.SfError, match="rows must be"):
        native.sf_bench_l2_gather_rate(3, 8, buf, 0, sink)

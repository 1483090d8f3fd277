"""The shared-memory gather-rate probe (the projector kernels' second roof) runs and rejects bad arguments (GPU)."""

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

"""The C-ABI library builds, loads and exports every declared symbol (CPU only).

Also checks the host-side argument validation that runs before any CUDA
call, so it can be exercised without a GPU.
"""

import ctypes
import os
import re

import pytest

from layer_optimizer_gb300 import build, native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return native.load()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(inc, f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                             src, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_lists_binding_exports():
    assert _declared() == set(native.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert native.sf_version() == "0.1.0"


def test_validation_errors_without_gpu(lib):
    hp = native.hparams()
    t = native.sf_tensor(16, 32, 64, 128, None, 10)
    arr = (native.sf_tensor * 1)(t)
    # step < 1 and bad hyper-parameters are rejected before any CUDA call
    assert lib.sf_adamw_layer_step(arr, 1, ctypes.byref(hp), 0, None) == native.SF_ERR_INVALID
    assert "step" in native.sf_last_error()
    bad = native.hparams(lr=float("nan"))
    assert lib.sf_adamw_layer_step(arr, 1, ctypes.byref(bad), 1, None) == native.SF_ERR_INVALID
    assert lib.sf_adamw_layer_step(arr, -1, ctypes.byref(hp), 1, None) == native.SF_ERR_INVALID
    assert lib.sf_adamw_layer_step(None, 1, ctypes.byref(hp), 1, None) == native.SF_ERR_INVALID
    assert lib.sf_adamw_layer_step(arr, 1, None, 1, None) == native.SF_ERR_INVALID
    neg = (native.sf_tensor * 1)(native.sf_tensor(16, 32, 64, 128, None, -1))
    assert lib.sf_adamw_layer_step(neg, 1, ctypes.byref(hp), 1, None) == native.SF_ERR_INVALID
    betas = native.hparams(beta1=1.0)
    assert lib.sf_adamw_layer_step(arr, 1, ctypes.byref(betas), 1, None) == native.SF_ERR_INVALID
    # an empty layer is a no-op
    assert lib.sf_adamw_layer_step(arr, 0, ctypes.byref(hp), 1, None) == native.SF_OK
    # compressed step
    assert lib.lsp_adamw_compressed(None, None, None, None, 4, ctypes.byref(hp), 1, None) == native.SF_ERR_INVALID
    assert lib.lsp_adamw_compressed(None, None, None, None, 0, ctypes.byref(hp), 0, None) == native.SF_ERR_INVALID
    # window creation
    out = ctypes.c_void_p()
    assert lib.sf_window_create(0, None, 1, None, None, None, ctypes.byref(out)) == native.SF_ERR_INVALID
    assert lib.sf_slide_window_step(None, None, 0, None, 0, None, None) == native.SF_ERR_INVALID
    # projector queries on NULL
    assert lib.lsp_projector_rows(None) == -1 and lib.lsp_projector_dim(None) == -1


def test_workspace_sizes_without_gpu(lib):
    # the workspace queries are host arithmetic on the shapes
    a = native.lsp_workspace_bytes(4096, 4096, 512)
    b = native.lsp_workspace_bytes(4096, 11008, 512)
    assert 4096 * 512 * 4 <= a < b                    # at least R^T (n x d fp32)
    f = native.lsp_fit_workspace_bytes(4096, 4096, 512, native.SF_FP32)
    assert f > a + 4096 * 4096 * 4                    # the compress pair's workspace plus G^T
    l1 = native.lce_workspace_bytes(8192, 4096, 128256, 4608)
    assert l1 == native.lce_workspace_bytes(8192, 64, 128256, 4608)   # nothing depends on D
    assert l1 >= 4608 * 128256 * (4 + 2)             # one chunk of fp32 logits and bf16 gradient
    # the chunk is clamped to the token count (rounded up to 8)
    assert native.lce_workspace_bytes(100, 64, 1000, 4096) == native.lce_workspace_bytes(100, 64, 1000, 104)
    assert native.lce_workspace_bytes(0, 64, 1000, 64) == 0


def test_gemm_probe_and_cross_entropy_validation_without_gpu(lib):
    # argument checks that return before any CUDA call
    f = ctypes.c_float(1.0)
    assert lib.sf_gemm_bf16(None, 0, None, 0, None, 1, 1, 1, 1, 1, 1, f, 0, None) == native.SF_ERR_INVALID
    assert lib.sf_gemm_bf16(16, 2, 16, 0, 16, 8, 8, 8, 8, 8, 8, f, 0, None) == native.SF_ERR_INVALID
    assert "layout" in native.sf_last_error()
    assert lib.sf_gemm_abt_bf16(16, 16, 16, 0, 8, 8, 8, 8, 8, f, 0, None) == native.SF_ERR_INVALID
    assert lib.sf_bench_gather_rate(0, 8, 16, None) == native.SF_ERR_INVALID
    loss = ctypes.c_double()
    assert lib.lce_forward_backward(None, 16, 16, 8, 8, 8, 8, -100, ctypes.byref(loss), None, None, 16, 1 << 20,
                                    None) == native.SF_ERR_INVALID
    assert lib.lce_forward_backward(16, 16, 16, 8, 8, 8, 12, -100, ctypes.byref(loss), None, None, 16, 1 << 20,
                                    None) == native.SF_ERR_INVALID       # chunk not a multiple of 8

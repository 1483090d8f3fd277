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

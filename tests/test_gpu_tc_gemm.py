"""Tensor-core GEMM C = alpha A B^T (+ C) against an fp64 product (GPU).

bf16 inputs, so every product is exact in fp32; the kernel sums K of them
in fp32, which the check bounds by 1e-5 of sum |a||b| per element.  The
shapes take the pair kernel through its edges: rows or columns that end
inside the second CTA's half of a 256 x 256 tile (or before it), ragged K,
and more tiles than CTA pairs.
"""

import numpy as np
import pytest
import torch

from _util import f64
from layer_optimizer_gb300 import native, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_GEMM = 1e-5


def _inputs(M, N, K, seed):
    A = synth.normal((M, K), 1.0, seed, dtype=torch.bfloat16)
    B = synth.normal((N, K), 1.0, seed + 1, dtype=torch.bfloat16)
    return A, B


def _check(C, A64, B64, C0=None, alpha=1.0):
    ref = alpha * (A64 @ B64.T)
    mag = abs(alpha) * (np.abs(A64) @ np.abs(B64).T)
    if C0 is not None:
        ref = ref + C0
        mag = mag + np.abs(C0)
    err = np.abs(f64(C) - ref)
    bad = err > TOL_GEMM * mag + 1e-30
    assert not bad.any(), (int(bad.sum()), float((err / (mag + 1e-30)).max()))


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 1024), (200, 300, 136), (1000, 777, 520),
                                   (64, 40, 8),          # the second CTA of the pair holds no row of A or B
                                   (384, 1024, 4096),    # odd number of 128-row halves
                                   (1, 1, 8), (129, 257, 72),
                                   (2000, 300, 64),      # more rows than columns: tiles taken n fastest
                                   (300, 5000, 256),
                                   (1500, 7000, 96)])    # 168 tiles: up to three per CTA pair, both accumulators reused
def test_gemm_matches_fp64(M, N, K):
    A, B = _inputs(M, N, K, M + N + K)
    C = torch.full((M, N), float("nan"), device=DEV)
    native.sf_gemm_abt_bf16(A.to(DEV), B.to(DEV), C, M, N, K, K, K, N)
    torch.cuda.synchronize()
    native.sf_sync_status()
    _check(C, f64(A), f64(B))


def test_gemm_accumulate_alpha_and_strides():
    M, N, K = 300, 520, 200
    A, B = _inputs(M, N, K, 7)
    lda, ldb, ldc = 208, 216, 528                 # padded rows
    Ad = torch.zeros(M, lda, dtype=torch.bfloat16, device=DEV)
    Bd = torch.zeros(N, ldb, dtype=torch.bfloat16, device=DEV)
    Ad[:, :K] = A.to(DEV)
    Bd[:, :K] = B.to(DEV)
    C0 = synth.normal((M, ldc), 1.0, 9).to(DEV)
    C = C0.clone()
    native.sf_gemm_abt_bf16(Ad, Bd, C, M, N, K, lda, ldb, ldc, alpha=-0.5, accumulate=True)
    torch.cuda.synchronize()
    _check(C[:, :N], f64(A), f64(B), C0=f64(C0[:, :N]), alpha=-0.5)
    assert torch.equal(C[:, N:], C0[:, N:])       # columns past N untouched


def test_gemm_is_deterministic_and_rejects_bad_strides():
    M, N, K = 256, 512, 512
    A, B = _inputs(M, N, K, 3)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C1, C2 = torch.empty(M, N, device=DEV), torch.empty(M, N, device=DEV)
    native.sf_gemm_abt_bf16(Ad, Bd, C1, M, N, K, K, K, N)
    native.sf_gemm_abt_bf16(Ad, Bd, C2, M, N, K, K, K, N)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    with pytest.raises(native.SfError, match="aligned"):
        native.sf_gemm_abt_bf16(Ad, Bd, C1, M, N, K - 4, K - 4, K, N)


@pytest.mark.parametrize("a_layout,b_layout", [(0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (64, 40, 8), (129, 257, 72), (2000, 300, 136),
                                   (1500, 7000, 96),
                                   # M, N multiples of 64: transposed operands load as one 3D box
                                   (384, 1024, 200), (1024, 640, 72), (2048, 4096, 320)])
def test_gemm_transposed_layouts(a_layout, b_layout, M, N, K):
    # an operand stored transposed (MN-major: [K][M] or [K][N]) with padded
    # rows; the product is the same as with both operands K-major
    A, B = _inputs(M, N, K, 31 + M + N + K)
    lda = -(-(M if a_layout else K) // 8) * 8 + 8       # rows padded, 16-byte multiples
    ldb = -(-(N if b_layout else K) // 8) * 8 + 16
    As = A.t() if a_layout else A
    Bs = B.t() if b_layout else B
    Ad = torch.zeros(As.shape[0], lda, dtype=torch.bfloat16, device=DEV)
    Bd = torch.zeros(Bs.shape[0], ldb, dtype=torch.bfloat16, device=DEV)
    Ad[:, :As.shape[1]] = As.to(DEV)
    Bd[:, :Bs.shape[1]] = Bs.to(DEV)
    C = torch.full((M, N), float("nan"), device=DEV)
    native.sf_gemm_bf16(Ad, a_layout, Bd, b_layout, C, M, N, K, lda, ldb, N)
    torch.cuda.synchronize()
    native.sf_sync_status()
    _check(C, f64(A), f64(B))
    C0 = C.clone()
    native.sf_gemm_bf16(Ad, a_layout, Bd, b_layout, C, M, N, K, lda, ldb, N, alpha=2.0, accumulate=True)
    torch.cuda.synchronize()
    _check(C, f64(A), f64(B), C0=f64(C0), alpha=2.0)


def test_gemm_layout_rejections():
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    C = torch.empty(64, 64, device=DEV)
    with pytest.raises(native.SfError, match="layout"):
        native.sf_gemm_bf16(A, 2, A, 0, C, 64, 64, 64, 64, 64, 64)
    with pytest.raises(native.SfError, match="leading"):
        native.sf_gemm_bf16(A, 1, A, 0, C, 72, 64, 64, 64, 64, 64)     # lda 64 < M 72 for a transposed A

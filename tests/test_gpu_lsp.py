"""Parity of the sparse-projector path with the fp64 oracle (GPU).

Covers the bookkeeping (bit-exact), compress (the TMA-staged gather, the
plain-load path, a gradient in pinned host memory), the compressed AdamW step, and decompress-apply into fp32
(with bf16 mirror) and bf16 weights, on shapes that span several tiles and
ragged tails, plus the full LLaMA-7B projector workload.
"""

import numpy as np
import pytest
import torch

from _util import HP, TOL_LSP, TOL_STATE, bits, check_bf16_applied, check_close, f64
from layer_optimizer_gb300 import native, synth
from oracle import adamw as oa
from oracle import bf16 as ob
from oracle import lsp as ol

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _make(rows, d, k, seed):
    idx, val = synth.projector(rows, d, k, seed)
    h = native.lsp_projector_create(rows, d, k, torch.from_numpy(idx).to(DEV), torch.from_numpy(val).to(DEV))
    return h, ol.Projector(idx, val, d)


def _ws(m, n, d):
    nb = native.lsp_workspace_bytes(m, n, d)
    return torch.empty(max(nb, 256), dtype=torch.uint8, device=DEV), nb


# ---------------------------------------------------------------- bookkeeping

@pytest.mark.parametrize("rows,d,k", [(1, 1, 1), (37, 8, 3), (1024, 64, 4), (4096, 512, 8), (11008, 512, 8),
                                      (200, 12, 5), (130, 1024, 2), (100, 128, 64)])
def test_bookkeeping_bit_exact(rows, d, k):
    h, ref = _make(rows, d, k, rows + d)
    cp = torch.empty(d + 1, dtype=torch.int32, device=DEV)
    ri = torch.empty(rows * k, dtype=torch.int32, device=DEV)
    cv = torch.empty(rows * k, dtype=torch.float32, device=DEV)
    bp = torch.empty(d, dtype=torch.int32, device=DEV)
    native.lsp_projector_export_csc(h, cp, ri, cv, bp)
    torch.cuda.synchronize()
    col_ptr, row_idx, val = ol.ell_to_csc(ref)
    assert np.array_equal(cp.cpu().numpy(), col_ptr)
    assert np.array_equal(ri.cpu().numpy(), row_idx)
    assert np.array_equal(cv.cpu().numpy().view(np.uint32), val.astype(np.float32).view(np.uint32))
    assert np.array_equal(bp.cpu().numpy(), ol.bucket_perm(col_ptr))
    assert (h.rows, h.d, h.k) == (rows, d, k)


def test_validation_rejects_bad_ids():
    idx, val = synth.projector(50, 16, 3, 1)
    bad = idx.copy()
    bad[7, 1] = bad[7, 0]                      # repeated id in a row
    with pytest.raises(native.SfError, match="repeats"):
        native.lsp_projector_create(50, 16, 3, torch.from_numpy(bad).to(DEV), torch.from_numpy(val).to(DEV))
    bad = idx.copy()
    bad[3, 2] = 16                             # out of range
    with pytest.raises(native.SfError, match="outside"):
        native.lsp_projector_create(50, 16, 3, torch.from_numpy(bad).to(DEV), torch.from_numpy(val).to(DEV))
    with pytest.raises(native.SfError):
        native.lsp_projector_create(50, 0, 3, torch.from_numpy(idx).to(DEV), torch.from_numpy(val).to(DEV))


# ------------------------------------------------------------------ compress

COMPRESS_CASES = [
    # (m, n, d, k, dtype)   -- TMA path needs n * elem_size % 16 == 0
    (1, 1, 1, 1, torch.float32),          # generic
    (7, 33, 8, 2, torch.float32),         # generic (n * 4 not a multiple of 16)
    (33, 7, 16, 16, torch.bfloat16),      # generic, k = d
    (64, 128, 16, 2, torch.float32),
    (100, 128, 8, 3, torch.float32),      # ragged rows (window tail)
    (1000, 1000, 64, 4, torch.float32),   # ragged rows and columns, row splits
    (1024, 1024, 64, 4, torch.bfloat16),  # the one-linear-layer workload
    (333, 264, 512, 8, torch.float32),    # d = 512: 4 ranges of 128 outputs (32 warps each)
    (260, 136, 200, 3, torch.bfloat16),   # d = 200: a full and a ragged output range
    (150, 96, 300, 5, torch.float32),     # d = 300: 3 output ranges
    (129, 64, 12, 3, torch.float32),      # d not a multiple of 8
    (50, 40, 30, 3, torch.float32),       # d not a multiple of 4: stage 2 as the staged gather
    (300, 5000, 512, 8, torch.float32),   # 160 tiles: one whole wave, 2 column blocks split 3 ways (ragged last)
    (700, 9800, 256, 4, torch.bfloat16),  # 154 tiles: one whole wave, 1 ragged column block split 6 ways
    (300, 264, 1024, 8, torch.float32),   # d at its maximum: 8 output ranges
    (200, 160, 128, 64, torch.float32),   # k at its maximum: slices too large for the ring, plain loads
    (150, 136, 64, 32, torch.bfloat16),   # k = 32
]


@pytest.mark.parametrize("m,n,d,k,dt", [(333, 264, 512, 8, torch.float32), (1024, 1024, 64, 4, torch.bfloat16)])
def test_compress_reads_pinned_host_gradient_with_plain_loads(m, n, d, k, dt):
    # tensor maps address only this device's memory: a G in pinned host
    # memory takes the plain-load gather over the host link, same result
    P, Pr = _make(m, d, k, 40 + m)
    Q, Qr = _make(n, d, k, 50 + n)
    G = synth.normal((m, n), 1e-3, 60 + m + n, dtype=dt).pin_memory()
    S = torch.full((d, d), float("nan"), device=DEV)
    ws, nb = _ws(m, n, d)
    native.lsp_compress(P, Q, G, native.SF_FP32 if dt == torch.float32 else native.SF_BF16, m, n, S, ws, nb)
    torch.cuda.synchronize()
    native.sf_sync_status()
    S_ref, S_abs = ol.compress(Pr, Qr, f64(G.float()))
    check_close("S (pinned host G)", S, S_ref, S_abs, TOL_LSP)


@pytest.mark.parametrize("m,n,d,k,dt", COMPRESS_CASES)
def test_compress_parity(m, n, d, k, dt):
    P, Pr = _make(m, d, k, 10 + m)
    Q, Qr = _make(n, d, k, 20 + n)
    G = synth.normal((m, n), 1e-3, 30 + m + n, dtype=dt).to(DEV)
    S = torch.full((d, d), float("nan"), device=DEV)
    ws, nb = _ws(m, n, d)
    native.lsp_compress(P, Q, G, native.SF_FP32 if dt == torch.float32 else native.SF_BF16, m, n, S, ws, nb)
    torch.cuda.synchronize()
    S_ref, S_abs = ol.compress(Pr, Qr, f64(G.float()))
    check_close("S", S, S_ref, S_abs, TOL_LSP)


def test_compress_deterministic_and_guarded():
    m, n, d, k = 700, 512, 512, 8
    P, _ = _make(m, d, k, 1)
    Q, _ = _make(n, d, k, 2)
    G = synth.normal((m, n), 1e-3, 3).to(DEV)
    ws, nb = _ws(m, n, d)
    pad = 1024
    buf = torch.full((d * d + 2 * pad,), 777.0, device=DEV)
    S1 = buf[pad:pad + d * d]
    native.lsp_compress(P, Q, G, native.SF_FP32, m, n, S1, ws, nb)
    S2 = torch.empty(d * d, device=DEV)
    native.lsp_compress(P, Q, G, native.SF_FP32, m, n, S2, ws, nb)
    torch.cuda.synchronize()
    assert torch.equal(S1.view(torch.int32), S2.view(torch.int32))
    assert torch.all(buf[:pad] == 777.0) and torch.all(buf[pad + d * d:] == 777.0)
    native.sf_sync_status()


def test_compress_rejects_bad_arguments():
    P, _ = _make(64, 16, 2, 1)
    Q, _ = _make(128, 16, 2, 2)
    Q8, _ = _make(128, 8, 2, 3)
    G = torch.zeros(64, 128, device=DEV)
    S = torch.zeros(16, 16, device=DEV)
    ws, nb = _ws(64, 128, 16)
    with pytest.raises(native.SfError, match="rows"):
        native.lsp_compress(P, Q, G, native.SF_FP32, 65, 128, S, ws, nb)
    with pytest.raises(native.SfError, match="differ"):
        native.lsp_compress(P, Q8, G, native.SF_FP32, 64, 128, S, ws, nb)
    with pytest.raises(native.SfError, match="workspace"):
        native.lsp_compress(P, Q, G, native.SF_FP32, 64, 128, S, ws, 16)


# ----------------------------------------------------- compressed AdamW step

def test_compressed_adamw_three_steps():
    d = 512
    S_seq = [synth.normal((d, d), 1e-4, 40 + t).to(DEV) for t in range(3)]
    m = torch.zeros(d, d, device=DEV)
    v = torch.zeros(d, d, device=DEV)
    dS = torch.empty(d, d, device=DEV)
    hp = native.hparams(**HP)
    for t in (1, 2, 3):
        m0, v0 = f64(m), f64(v)
        m_abs = np.abs(m0)
        native.lsp_adamw_compressed(S_seq[t - 1], m, v, dS, d * d, hp, t)
        torch.cuda.synchronize()
        ref, m_ref, v_ref, dS_abs, m_abs_new = oa.compressed_adamw_step(
            f64(S_seq[t - 1]), m0, v0, t, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], m_abs)
        check_close("m", m, m_ref, m_abs_new, TOL_STATE)
        check_close("v", v, v_ref, v_ref, TOL_STATE)
        check_close("dS", dS, ref, dS_abs, TOL_STATE)


# ---------------------------------------------------------------- decompress

DECOMPRESS_CASES = [
    (1, 1, 1, 1), (7, 33, 8, 2), (64, 128, 16, 2), (100, 130, 8, 3), (1000, 1000, 64, 4),
    (333, 264, 512, 8), (129, 63, 12, 3), (40, 50, 600, 4),   # d > 512: generic path
    (64, 96, 64, 16), (100, 72, 40, 12),                       # k > 8: generic V, fast apply
    (96, 520, 64, 8), (200, 136, 128, 8),                      # V as row gathers of dS^T (k = 8, d % 64 = 0)
    (100, 132, 64, 8),                                         # k = 8 but n % 8 != 0: V from the staged block
    (100, 72, 1024, 8),                                        # d at its maximum: generic path
    (80, 96, 128, 64),                                         # k at its maximum: generic V and apply
    (90, 70, 64, 32),                                          # k = 32: fast apply, one row per group
]


@pytest.mark.parametrize("m,n,d,k", DECOMPRESS_CASES)
@pytest.mark.parametrize("wtype", ["fp32", "fp32+mirror", "bf16"])
def test_decompress_apply_parity(m, n, d, k, wtype):
    P, Pr = _make(m, d, k, 50 + m)
    Q, Qr = _make(n, d, k, 60 + n)
    dS = synth.normal((d, d), 1e-4, 70 + d).to(DEV)
    W0 = synth.normal((m, n), 0.02, 80 + m)
    ws, nb = _ws(m, n, d)
    D, D_abs = ol.decompress(Pr, Qr, f64(dS))
    if wtype == "bf16":
        W = W0.to(torch.bfloat16).to(DEV)
        wb0 = bits(W)
        native.lsp_decompress_apply(P, Q, dS, W, native.SF_BF16, None, m, n, ws, nb)
        torch.cuda.synchronize()
        check_bf16_applied("W bf16", bits(W), ob.bits_to_f64(wb0), D, D_abs)
    else:
        W = W0.to(DEV)
        mirror = torch.empty(m, n, dtype=torch.bfloat16, device=DEV) if wtype.endswith("mirror") else None
        native.lsp_decompress_apply(P, Q, dS, W, native.SF_FP32, mirror, m, n, ws, nb)
        torch.cuda.synchronize()
        W_ref = ol.apply_fp32(f64(W0), D)
        # error budget: fp32 rounding of D (relative to its magnitude) plus one rounding of W - D
        err = np.abs(f64(W) - W_ref)
        assert np.all(err <= TOL_LSP * D_abs + 2.0 ** -23 * np.abs(W_ref) + 1e-30), float(err.max())
        if mirror is not None:
            assert np.array_equal(bits(mirror), ob.bf16_bits(f64(W)))


def test_apply_in_place_deterministic():
    m, n, d, k = 300, 256, 512, 8
    P, _ = _make(m, d, k, 1)
    Q, _ = _make(n, d, k, 2)
    dS = synth.normal((d, d), 1e-4, 3).to(DEV)
    W0 = synth.normal((m, n), 0.02, 4).to(DEV)
    ws, nb = _ws(m, n, d)
    Wa, Wb = W0.clone(), W0.clone()
    native.lsp_decompress_apply(P, Q, dS, Wa, native.SF_FP32, None, m, n, ws, nb)
    native.lsp_decompress_apply(P, Q, dS, Wb, native.SF_FP32, None, m, n, ws, nb)
    torch.cuda.synchronize()
    assert torch.equal(Wa.view(torch.int32), Wb.view(torch.int32))


# --------------------------------------------------- chained workloads

def test_one_linear_layer_chain_three_steps():
    """W 1024 x 1024 fp32 master, bf16 G, d = 64, k = 4, 3 steps of the chain."""
    m = n = 1024
    d, k = 64, 4
    P, Pr = _make(m, d, k, 101)
    Q, Qr = _make(n, d, k, 102)
    W = synth.normal((m, n), 0.02, 0).to(DEV)
    mirror = torch.empty(m, n, dtype=torch.bfloat16, device=DEV)
    mm = torch.zeros(d, d, device=DEV)
    vv = torch.zeros(d, d, device=DEV)
    S = torch.empty(d, d, device=DEV)
    dS = torch.empty(d, d, device=DEV)
    ws, nb = _ws(m, n, d)
    hp = native.hparams(**HP)
    for t in (1, 2, 3):
        G = synth.normal((m, n), 1e-3, synth.sub_seed(0, 1, 0, t), dtype=torch.bfloat16).to(DEV)
        W_in = f64(W)
        m0, v0 = f64(mm), f64(vv)
        native.lsp_compress(P, Q, G, native.SF_BF16, m, n, S, ws, nb)
        native.lsp_adamw_compressed(S, mm, vv, dS, d * d, hp, t)
        native.lsp_decompress_apply(P, Q, dS, W, native.SF_FP32, mirror, m, n, ws, nb)
        torch.cuda.synchronize()
        S_ref, S_abs = ol.compress(Pr, Qr, f64(G.float()))
        check_close(f"S t={t}", S, S_ref, S_abs, TOL_LSP)
        dS_ref, _, _, dS_abs, _ = oa.compressed_adamw_step(f64(S), m0, v0, t, HP["lr"], HP["beta1"],
                                                           HP["beta2"], HP["eps"])
        check_close(f"dS t={t}", dS, dS_ref, dS_abs, TOL_STATE)
        D, D_abs = ol.decompress(Pr, Qr, f64(dS))
        err = np.abs(f64(W) - (W_in - D))
        assert np.all(err <= TOL_LSP * D_abs + 2.0 ** -23 * np.abs(W_in - D)), float(err.max())
        assert np.array_equal(bits(mirror), ob.bf16_bits(f64(W)))


@pytest.mark.slow
def test_llama7b_matrices_full_size():
    """q, k, v, o, gate, up, down: G fp32, W bf16, d = 512, k = 8, one step; exhaustive parity."""
    d, k = 512, 8
    hp = native.hparams(**HP)
    for mi, (name, m, n) in enumerate(synth.LLAMA7_LSP_MATRICES):
        if name in ("k", "v"):      # same shape as q; covered
            continue
        Pi, Pv = synth.projector(m, d, k, synth.sub_seed(7, mi, 0))
        Qi, Qv = synth.projector(n, d, k, synth.sub_seed(7, mi, 1))
        P = native.lsp_projector_create(m, d, k, torch.from_numpy(Pi).to(DEV), torch.from_numpy(Pv).to(DEV))
        Q = native.lsp_projector_create(n, d, k, torch.from_numpy(Qi).to(DEV), torch.from_numpy(Qv).to(DEV))
        Pr, Qr = ol.Projector(Pi, Pv, d), ol.Projector(Qi, Qv, d)
        G = synth.fill_normal_(torch.empty(m, n, device=DEV), 1e-3, synth.sub_seed(8, mi))
        W = synth.fill_normal_(torch.empty(m, n, dtype=torch.bfloat16, device=DEV), 0.02, synth.sub_seed(9, mi))
        wb0 = bits(W)
        S = torch.empty(d, d, device=DEV)
        mm, vv, dS = (torch.zeros(d, d, device=DEV) for _ in range(3))
        ws, nb = _ws(m, n, d)
        native.lsp_compress(P, Q, G, native.SF_FP32, m, n, S, ws, nb)
        native.lsp_adamw_compressed(S, mm, vv, dS, d * d, hp, 1)
        native.lsp_decompress_apply(P, Q, dS, W, native.SF_BF16, None, m, n, ws, nb)
        torch.cuda.synchronize()
        S_ref, S_abs = ol.compress(Pr, Qr, f64(G))
        check_close(f"S {name}", S, S_ref, S_abs, TOL_LSP)
        D, D_abs = ol.decompress(Pr, Qr, f64(dS))
        check_bf16_applied(f"W {name}", bits(W), ob.bits_to_f64(wb0), D, D_abs)
        del G, W, ws
        torch.cuda.empty_cache()

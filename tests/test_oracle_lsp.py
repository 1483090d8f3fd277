"""Pins for the fp64 learned-sparse-projector oracle (CPU only).

Compress is pinned by brute-force sums on tiny shapes, by the k = d dense
case, by a permutation projector, and by linearity; decompress by the
adjoint identity and by orthonormal projectors; the bookkeeping by scipy's
CSR -> CSC conversion and by structural invariants.
"""

import numpy as np
import pytest
import scipy.sparse as sp

from layer_optimizer_gb300 import synth
from oracle import lsp as ol


def _proj(rows, d, k, seed, replace=False):
    idx, val = synth.projector(rows, d, k, seed, replace=replace)
    return ol.Projector(idx, val, d)


def _brute_compress(P, Q, G):
    m, n = G.shape
    S = np.zeros((P.d, Q.d))
    for i in range(m):
        for li in range(P.k):
            a, p = P.idx[i, li], P.val[i, li]
            for j in range(n):
                for lj in range(Q.k):
                    S[a, Q.idx[j, lj]] += p * G[i, j] * Q.val[j, lj]
    return S


@pytest.mark.parametrize("m,n,d,k", [
    (1, 1, 1, 1), (7, 33, 8, 2), (33, 7, 8, 1), (64, 100, 16, 2), (100, 64, 16, 16),
    (7, 7, 8, 8), (33, 33, 16, 1),
])
def test_compress_brute_force(m, n, d, k):
    rng = np.random.default_rng(m * 1000 + n)
    G = rng.standard_normal((m, n))
    P, Q = _proj(m, d, k, 1), _proj(n, d, k, 2)
    S, S_abs = ol.compress(P, Q, G)
    Sb = _brute_compress(P, Q, G)
    np.testing.assert_allclose(S, Sb, rtol=1e-12, atol=1e-12)
    Sab = _brute_compress(ol.Projector(P.idx, np.abs(P.val), d),
                          ol.Projector(Q.idx, np.abs(Q.val), d), np.abs(G))
    np.testing.assert_allclose(S_abs, Sab, rtol=1e-12, atol=1e-12)


def test_compress_dense_special_case():
    # k = d with ids 0..d-1 in every row: P and Q are dense, and S is the
    # ordinary product written as explicit sums.
    rng = np.random.default_rng(5)
    m, n, d = 9, 11, 4
    Pd, Qd, G = rng.standard_normal((m, d)), rng.standard_normal((n, d)), rng.standard_normal((m, n))
    P = ol.Projector(np.tile(np.arange(d), (m, 1)), Pd, d)
    Q = ol.Projector(np.tile(np.arange(d)[::-1], (n, 1)), Qd[:, ::-1], d)
    S, _ = ol.compress(P, Q, G)
    want = np.array([[sum(Pd[i, a] * G[i, j] * Qd[j, c] for i in range(m) for j in range(n))
                      for c in range(d)] for a in range(d)])
    np.testing.assert_allclose(S, want, rtol=1e-12)


def test_compress_permutation_projector():
    # m = d, k = 1, value 1: P^T permutes rows, so S[pi(i)] = (G Q)[i].
    rng = np.random.default_rng(6)
    d, n = 16, 40
    perm = rng.permutation(d)
    P = ol.Projector(perm[:, None], np.ones((d, 1)), d)
    Q = _proj(n, d, 3, 7)
    G = rng.standard_normal((d, n))
    S, _ = ol.compress(P, Q, G)
    GQ = np.array([[sum(G[i, j] * Q.val[j, l] for j in range(n) for l in range(Q.k) if Q.idx[j, l] == c)
                    for c in range(d)] for i in range(d)])
    np.testing.assert_allclose(S[perm], GQ, rtol=1e-12, atol=1e-14)


def test_compress_linearity():
    rng = np.random.default_rng(8)
    P, Q = _proj(50, 16, 4, 1), _proj(70, 16, 4, 2)
    G1, G2 = rng.standard_normal((50, 70)), rng.standard_normal((50, 70))
    a, b = 0.37, -2.5
    lhs, _ = ol.compress(P, Q, a * G1 + b * G2)
    s1, _ = ol.compress(P, Q, G1)
    s2, _ = ol.compress(P, Q, G2)
    np.testing.assert_allclose(lhs, a * s1 + b * s2, rtol=1e-11, atol=1e-12)


def test_adjoint_identity():
    # <P^T G Q, X>_F = <G, P X Q^T>_F: compress and decompress are adjoint maps.
    rng = np.random.default_rng(9)
    P, Q = _proj(40, 8, 3, 3), _proj(30, 8, 3, 4)
    G, X = rng.standard_normal((40, 30)), rng.standard_normal((8, 8))
    S, _ = ol.compress(P, Q, G)
    D, _ = ol.decompress(P, Q, X)
    assert np.sum(S * X) == pytest.approx(np.sum(G * D), rel=1e-12)


def test_round_trip_identity():
    # decompress(compress(G)) = P P^T G Q Q^T, with the products spelled out
    # as sums over the ELL lists.
    rng = np.random.default_rng(10)
    P, Q = _proj(12, 6, 2, 5), _proj(9, 6, 2, 6)
    G = rng.standard_normal((12, 9))
    S, _ = ol.compress(P, Q, G)
    D, _ = ol.decompress(P, Q, S)

    def ppt(Pr, rows):
        M = np.zeros((rows, rows))
        for i in range(rows):
            for i2 in range(rows):
                M[i, i2] = sum(Pr.val[i, l] * Pr.val[i2, l2] for l in range(Pr.k) for l2 in range(Pr.k)
                               if Pr.idx[i, l] == Pr.idx[i2, l2])
        return M
    want = ppt(P, 12) @ G @ ppt(Q, 9)
    np.testing.assert_allclose(D, want, rtol=1e-11, atol=1e-12)


def test_orthonormal_projectors_invert():
    # Disjoint supports with values 1/sqrt(count) give P^T P = I, so
    # compress(decompress(X)) = X.
    d, per = 8, 3
    rows = d * per
    idx = np.repeat(np.arange(d), per)[np.random.default_rng(1).permutation(rows)][:, None]
    val = np.full((rows, 1), 1 / np.sqrt(per))
    P = Q = ol.Projector(idx, val, d)
    X = np.random.default_rng(2).standard_normal((d, d))
    D, _ = ol.decompress(P, Q, X)
    S, _ = ol.compress(P, Q, D)
    np.testing.assert_allclose(S, X, rtol=1e-12, atol=1e-13)


def test_decompress_magnitude_and_apply():
    rng = np.random.default_rng(11)
    P, Q = _proj(20, 8, 2, 1), _proj(25, 8, 2, 2)
    X = rng.standard_normal((8, 8))
    D, D_abs = ol.decompress(P, Q, X)
    assert np.all(D_abs >= np.abs(D) * (1 - 1e-14))
    W = rng.standard_normal((20, 25))
    np.testing.assert_allclose(ol.apply_fp32(W, D), W - D)
    from oracle.bf16 import bf16_bits, bits_to_f64
    wb = bf16_bits(W)
    out = ol.apply_bf16(wb, D)
    np.testing.assert_array_equal(out, bf16_bits(bits_to_f64(wb) - D))


# ------------------------------------------------------------ bookkeeping --

@pytest.mark.parametrize("rows,d,k,replace", [(1, 1, 1, False), (37, 8, 3, False), (1024, 64, 4, False),
                                              (300, 16, 5, True), (50, 512, 8, False)])
def test_csc_matches_scipy_and_invariants(rows, d, k, replace):
    P = _proj(rows, d, k, 3, replace=replace)
    col_ptr, row_idx, val = ol.ell_to_csc(P)
    assert col_ptr[0] == 0 and col_ptr[-1] == rows * k
    assert np.all(np.diff(col_ptr) >= 0)
    for c in range(d):
        r = row_idx[col_ptr[c]:col_ptr[c + 1]]
        assert np.all(np.diff(r) >= 0), "rows ascend within a column"
    # scipy: CSR (duplicates kept, in slot order) -> CSC with sorted indices
    csr = sp.csr_matrix((P.val.ravel(), P.idx.ravel(), np.arange(0, rows * k + 1, k)), shape=(rows, d))
    if not replace:
        csc = csr.tocsc()
        csc.sort_indices()
        np.testing.assert_array_equal(col_ptr, csc.indptr)
        np.testing.assert_array_equal(row_idx, csc.indices)
        np.testing.assert_array_equal(val, csc.data)
    # CSC -> ELL round trip: each row gets back its (id, value) multiset
    back = [[] for _ in range(rows)]
    for c in range(d):
        for e in range(col_ptr[c], col_ptr[c + 1]):
            back[row_idx[e]].append((c, val[e]))
    for i in range(rows):
        assert sorted(back[i]) == sorted(zip(P.idx[i].tolist(), P.val[i].tolist()))


def test_nnz_bucket_values():
    want = {0: 0, 1: 1, 2: 2, 3: 3, 4: 3, 5: 4, 8: 4, 9: 5, 64: 7, 65: 8, 172: 9}
    for nnz, b in want.items():
        assert ol.nnz_bucket(nnz) == b


def test_bucket_perm_order():
    P = _proj(700, 64, 3, 4)
    col_ptr, _, _ = ol.ell_to_csc(P)
    perm = ol.bucket_perm(col_ptr)
    assert sorted(perm.tolist()) == list(range(64))
    keys = [(ol.nnz_bucket(col_ptr[c + 1] - col_ptr[c]), c) for c in perm]
    assert keys == sorted(keys)
    # an empty column sorts first
    idx = np.array([[1], [1], [2]])
    P2 = ol.Projector(idx, np.ones((3, 1)), 4)
    cp, _, _ = ol.ell_to_csc(P2)
    assert ol.bucket_perm(cp).tolist() == [0, 3, 2, 1]

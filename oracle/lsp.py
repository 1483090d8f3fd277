"""fp64 learned-sparse-projector path (test infrastructure only).

What it follows
---------------
"Practical offloading for fine-tuning LLM on commodity GPU via learned
sparse projectors" (abstract; method section "core idea" and "technical
framework"): the gradient that would cross the host link is compressed with
sparse projectors, the optimizer runs in the compressed space, and the
result is decompressed and applied on the GPU.  The pages give no formula;
the operation written out here is the plain reading of that description:

    S  = P^T . G . Q                     (m x n  ->  d x d)
    dS = compressed AdamW step on S      (see oracle.adamw)
    W <- W - P . dS . Q^T                (d x d  ->  m x n)

with P (m x d) and Q (n x d) sparse, holding a fixed number k of nonzeros in
every row ("sparse projectors", method section).

The projector bookkeeping is the transpose of the fixed-k-per-row layout
(ELL) into column lists (CSC) with rows ascending inside each column,
built by a stable counting sort, plus a column order grouped by list length
(nnz bucket = 0 for an empty column, else ceil(log2 nnz) + 1; columns in
ascending id inside a bucket).

Products use numpy matmul on dense fp64 copies of P and Q: the plain
definition of the triple product, one library primitive per product, no
blocking or reordering of our own.
"""

import numpy as np

from .bf16 import bf16_bits, bits_to_f64


class Projector:
    """A sparse projector with k nonzeros per row, stored as ELL.

    ``idx`` int array [rows, k] of column ids in [0, d), ``val`` float array
    [rows, k].  Values are widened to float64 exactly.
    """

    def __init__(self, idx, val, d):
        self.idx = np.asarray(idx, dtype=np.int64)
        self.val = np.asarray(val, dtype=np.float64)
        if self.idx.ndim != 2 or self.idx.shape != self.val.shape:
            raise ValueError("idx and val must both be [rows, k]")
        self.rows, self.k = self.idx.shape
        self.d = int(d)

    def dense(self):
        """Dense fp64 [rows, d] matrix; repeated ids in a row add up."""
        out = np.zeros((self.rows, self.d), dtype=np.float64)
        r = np.repeat(np.arange(self.rows), self.k)
        np.add.at(out, (r, self.idx.ravel()), self.val.ravel())
        return out


# ----------------------------------------------------------------------------
# Bookkeeping: ELL -> CSC of the same matrix, and the nnz-bucket column order
# ----------------------------------------------------------------------------

def ell_to_csc(proj):
    """Column lists of ``proj``: (col_ptr [d+1], row_idx [rows*k], val [rows*k]).

    Stable counting sort over the row-major ELL entries, so rows ascend
    within every column (and, for a repeated id in one row, the ELL slot
    order is kept).
    """
    d = proj.d
    flat_c = proj.idx.ravel()
    flat_r = np.repeat(np.arange(proj.rows, dtype=np.int64), proj.k)
    flat_v = proj.val.ravel()
    counts = np.zeros(d, dtype=np.int64)
    for c in flat_c:
        counts[c] += 1
    col_ptr = np.zeros(d + 1, dtype=np.int64)
    col_ptr[1:] = np.cumsum(counts)
    fill = col_ptr[:-1].copy()
    row_idx = np.empty(flat_c.size, dtype=np.int64)
    val = np.empty(flat_c.size, dtype=np.float64)
    for e in range(flat_c.size):          # entries visited in row-major order
        c = flat_c[e]
        row_idx[fill[c]] = flat_r[e]
        val[fill[c]] = flat_v[e]
        fill[c] += 1
    return col_ptr, row_idx, val


def nnz_bucket(nnz):
    """Bucket of a column list of length ``nnz``: 0 if empty, else ceil(log2 nnz)+1."""
    nnz = int(nnz)
    if nnz <= 0:
        return 0
    b = 0
    while (1 << b) < nnz:
        b += 1
    return b + 1


def bucket_perm(col_ptr):
    """Column ids ordered by (nnz bucket, column id)."""
    d = len(col_ptr) - 1
    keys = [(nnz_bucket(col_ptr[c + 1] - col_ptr[c]), c) for c in range(d)]
    return np.array([c for _, c in sorted(keys)], dtype=np.int64)


# ----------------------------------------------------------------------------
# Compress, decompress
# ----------------------------------------------------------------------------

def compress(P, Q, G):
    """S = P^T G Q and its magnitude |P|^T |G| |Q| (both fp64, d x d)."""
    G = np.asarray(G, dtype=np.float64)
    Pd, Qd = P.dense(), Q.dense()
    S = (Pd.T @ G) @ Qd
    S_abs = (np.abs(Pd).T @ np.abs(G)) @ np.abs(Qd)
    return S, S_abs


def decompress(P, Q, dS):
    """D = P dS Q^T and its magnitude |P| |dS| |Q|^T (fp64, m x n)."""
    dS = np.asarray(dS, dtype=np.float64)
    Pd, Qd = P.dense(), Q.dense()
    D = (Pd @ dS) @ Qd.T
    D_abs = (np.abs(Pd) @ np.abs(dS)) @ np.abs(Qd).T
    return D, D_abs


def apply_fp32(W, D):
    """W - D for an fp32 master held as fp64 values."""
    return np.asarray(W, dtype=np.float64) - D


def apply_bf16(W_bits, D):
    """RNE_bf16(W - D) for bf16 weights given as bit patterns."""
    return bf16_bits(bits_to_f64(W_bits) - D)

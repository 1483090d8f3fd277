// Learning the projectors: one gradient step on the stored values of P and
// Q for the reconstruction error of a gradient sample (LSP-Offload, method
// section, "key design": the sparse projectors are fitted by gradient
// descent to minimise what compressing and decompressing lose).
#include <cuda_bf16.h>

#include <algorithm>

#include "common.h"
#include "lsp_internal.cuh"
#include "ptx.cuh"

using sf::ceil_div;
using sf::fail;

// ----------------------------------------------------------------------------
// Projector fit step: one gradient step on the stored values of P and Q for
// L = ||G - P S Q^T||_F^2, S = P^T G Q.
// ----------------------------------------------------------------------------
// Written with E = G - P S Q^T, T = G Q, U = G^T P, A_P = P^T P, A_Q = Q^T Q:
//   E Q      = T - P (S A_Q)                    P^T E Q = S - A_P S A_Q = C
//   dL/dP[i,a] = -2 ( <T[i,:], (S + C)[a,:]> - sum_t P[i,a_t] (S A_Q S^T)[a_t, a] )
//   dL/dQ[j,b] = -2 ( <U[j,:], (S + C)^T[b,:]> - sum_t Q[j,b_t] (S^T A_P S)[b_t, b] )
//   L = ||G||^2 - 2 ||S||^2 + <A_P S, S A_Q>
// so the m x n error E is never formed: the step needs the compress pair
// (U, then S), one more gather for T over G^T, the two d x d Gram matrices
// (from the sparse forms), five d x d products, and per-row dot products at
// the k stored positions.
namespace sf {
namespace {

// out[j][i] = in[i][j] (in m x n, out n x m) through a padded 64 x 64 tile
// (16 loads in flight per thread), with this block's sum of in^2 (fp32
// within the block, one double out).
template <typename TB>
__global__ void __launch_bounds__(256) k_transpose_sumsq(const TB* __restrict__ in, int64_t m, int64_t n,
                                                         TB* __restrict__ out, double* __restrict__ partial) {
  __shared__ TB tile[64][65];
  __shared__ float red[8];
  const int64_t i0 = (int64_t)blockIdx.y * 64, j0 = (int64_t)blockIdx.x * 64;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
  float sq = 0.0f;
#pragma unroll 4
  for (int r = ty; r < 64; r += 4) {
    const int64_t i = i0 + r, j = j0 + tx;
    if (i < m && j < n) {
      const TB v = in[i * n + j];
      tile[r][tx] = v;
      float f;
      if constexpr (sizeof(TB) == 4) f = v;
      else f = __bfloat162float(v);
      sq = fmaf(f, f, sq);
    }
  }
  __syncthreads();
#pragma unroll 4
  for (int r = ty; r < 64; r += 4) {
    const int64_t j = j0 + r, i = i0 + tx;
    if (j < n && i < m) out[j * m + i] = tile[tx][r];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sq;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.0f;
    for (int w = 0; w < 8; ++w) b += red[w];
    partial[(int64_t)blockIdx.y * gridDim.x + blockIdx.x] = (double)b;
  }
}

// Gram matrix A = X^T X of a projector X (rows x d, k entries per row),
// straight from its sparse form: row a of A is the sum, over the entries
// (i, v) of column a (rows ascending), of v times row i of X, i.e. of
// v * x_t at column id_t for the k entries (id_t, x_t) of row i.  Four
// warps per output row, each over a quarter of column a's entries into its
// own shared-memory row; the quarters are then added in order.  In a warp
// the lanes split into R = 32 / k row groups of k slots (one group of 32
// slots per pass when k > 32); each lane loads its (entry, slot) pair for
// kGramB batches of R rows at once (independent loads), then the rows are
// applied one after another: a row's slots hit distinct output columns, so
// its lanes add at once.  A batch in which some row repeats an id
// (possible without validation) is applied slot by slot by the lanes that
// own the output columns.  Every sum runs in a fixed order; m k^2
// multiply-adds in all instead of the m d k of a gather over a dense copy.
constexpr int kGramWarps = 8, kGramSplit = 4, kGramB = 8;
__global__ void __launch_bounds__(32 * kGramWarps) k_gram_sparse(const int32_t* __restrict__ col_ptr,
                                                                 const int32_t* __restrict__ row_idx,
                                                                 const float* __restrict__ csc_val,
                                                                 const int32_t* __restrict__ ell_idx,
                                                                 const float* __restrict__ ell_val, int k, int d,
                                                                 float* __restrict__ A) {
  extern __shared__ float gram_rows[];   // [kGramWarps][d]: one partial row per warp
  const unsigned kAll = 0xffffffffu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp % kGramSplit;
  const int a = blockIdx.x * (kGramWarps / kGramSplit) + warp / kGramSplit;
  float* rb = gram_rows + (size_t)warp * d;
  for (int c = lane; c < d; c += 32) rb[c] = 0.0f;
  __syncwarp();
  if (a < d) {
    const int S = k < 32 ? k : 32;       // slots per row group and pass
    const int R = 32 / S;                // rows per batch
    const int r_l = lane / S, t_l = lane % S;
    const int c0 = col_ptr[a], len = col_ptr[a + 1] - c0;
    const int e0 = c0 + (int)((int64_t)len * quarter / kGramSplit);
    const int e1 = c0 + (int)((int64_t)len * (quarter + 1) / kGramSplit);
    for (int eb0 = e0; eb0 < e1; eb0 += R * kGramB) {
      for (int t0 = 0; t0 < k; t0 += S) {
        int bq[kGramB];
        float vq[kGramB], xq[kGramB];
#pragma unroll
        for (int q = 0; q < kGramB; ++q) {
          const int e = eb0 + q * R + r_l, t = t0 + t_l;
          bq[q] = 0;
          vq[q] = 0.0f;
          xq[q] = 0.0f;
          if (r_l < R && e < e1 && t < k) {
            const int64_t i = row_idx[e];
            vq[q] = csc_val[e];
            bq[q] = ell_idx[i * k + t];
            xq[q] = ell_val[i * k + t];
          }
        }
#pragma unroll
        for (int q = 0; q < kGramB; ++q) {
          const int eq = eb0 + q * R;
          if (eq >= e1) break;           // uniform
          const bool on = r_l < R && eq + r_l < e1 && t0 + t_l < k;
          // a repeated id inside a row of this batch: same (row, id) key
          const unsigned on_mask = __ballot_sync(kAll, on);
          unsigned peers = 0;
          if (on) peers = __match_any_sync(on_mask, (r_l << 26) | bq[q]);
          if (!__any_sync(kAll, on && __popc(peers) > 1)) {
            for (int r = 0; r < R && eq + r < e1; ++r) {
              if (on && r_l == r) rb[bq[q]] = fmaf(vq[q], xq[q], rb[bq[q]]);
              __syncwarp();
            }
          } else {
            for (int j = 0; j < 32; ++j) {
              if (!((on_mask >> j) & 1u)) continue;   // uniform
              const int bj = __shfl_sync(kAll, bq[q], j);
              const float vj = __shfl_sync(kAll, vq[q], j), xj = __shfl_sync(kAll, xq[q], j);
              if (lane == (bj & 31)) rb[bj] = fmaf(vj, xj, rb[bj]);
              __syncwarp();
            }
          }
        }
      }
    }
  }
  __syncthreads();
  if (a < d && quarter == 0) {
    const float* p0 = rb;
    for (int c = lane; c < d; c += 32) {
      float s = p0[c];
#pragma unroll
      for (int h = 1; h < kGramSplit; ++h) s += p0[(size_t)h * d + c];
      A[(int64_t)a * d + c] = s;
    }
  }
}

// C = op(A) op(B) for d x d fp32 row-major matrices, op = identity or
// transpose; up to three independent products per launch (blockIdx.z).
// 64 x 64 output tile per block, 4 x 4 per thread; every output sums over
// l = 0 .. d-1 in order with one accumulator.
struct DdJob {
  const float* A;
  const float* B;
  float* C;
  int ta, tb;
};
struct DdBatch {
  DdJob job[3];
  int d;
};

__global__ void __launch_bounds__(256) k_gemm_dd(const __grid_constant__ DdBatch bt) {
  const DdJob J = bt.job[blockIdx.z];
  const int d = bt.d;
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.0f;
  for (int k0 = 0; k0 < d; k0 += 16) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int q = threadIdx.x + 256 * r;
      // op(A)[i][l]: along l for a plain A, along i for a transposed one
      int kk, ii;
      if (J.ta) { ii = q & 63; kk = q >> 6; } else { kk = q & 15; ii = q >> 4; }
      const int i = i0 + ii, l = k0 + kk;
      As[kk][ii] = (i < d && l < d) ? (J.ta ? J.A[(int64_t)l * d + i] : J.A[(int64_t)i * d + l]) : 0.0f;
      int kb, jj;
      if (J.tb) { kb = q & 15; jj = q >> 4; } else { jj = q & 63; kb = q >> 6; }
      const int j = j0 + jj, lb = k0 + kb;
      Bs[kb][jj] = (j < d && lb < d) ? (J.tb ? J.B[(int64_t)j * d + lb] : J.B[(int64_t)lb * d + j]) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = As[kk][ty + 16 * r];
#pragma unroll
      for (int c = 0; c < 4; ++c) b[c] = Bs[kk][tx + 16 * c];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = i0 + ty + 16 * r, j = j0 + tx + 16 * c;
      if (i < d && j < d) J.C[(int64_t)i * d + j] = acc[r][c];
    }
}

// The same products when d is a multiple of 64: a 64 x 64 output tile per
// block of 64 threads, 8 x 8 outputs per thread accumulated as packed fp32
// pairs (fma.rn.f32x2: the same bits as fmaf).  Thread (ty, tx) owns rows
// 4 ty + {0..3} and 32 + 4 ty + {0..3} and the same columns with tx, so each
// 16-byte shared load of a k-row of op(A) or op(B) by a warp falls in one
// wavefront.  The k-slab of 32 is staged k-major from 16-byte global loads
// (the next slab's loads in flight while the current one is used); an
// operand stored along k (plain A, transposed B) is loaded one row per
// thread and written transposed with scalar stores that hit 32 distinct
// banks.
//
// SPLIT > 1 (d a multiple of 32 SPLIT): the sum over l is cut into SPLIT
// equal parts, one per CTA of a cluster of SPLIT along x, so a d x d product
// runs SPLIT times the blocks.  Each CTA sums its part in order, parks its
// 64 x 64 partial tile in shared memory, and after a cluster barrier CTA r
// adds its 64 / SPLIT rows of the tile over the SPLIT partials in rank
// order, reading its peers' shared memory, then stores them.  With SPLIT = 1
// every output sums l = 0 .. d-1 in order with one accumulator, as
// k_gemm_dd does.
template <int SPLIT>
__global__ void __launch_bounds__(64) k_gemm_dd64(const __grid_constant__ DdBatch bt) {
  static_assert(64 % SPLIT == 0, "the tile rows split evenly over the cluster");
  const DdJob J = bt.job[blockIdx.z];
  const int d = bt.d;
  __shared__ __align__(16) float As[32][64];
  __shared__ __align__(16) float Bs[32][64];
  const int tid = threadIdx.x, tx = tid & 7, ty = tid >> 3;
  const int i0 = blockIdx.y * 64, j0 = (blockIdx.x / SPLIT) * 64;
  const int part = d / SPLIT, l0 = (int)(blockIdx.x % SPLIT) * part;
  float4 ra[8], rb[8];
  // stored along k: thread t reads row t of the slab (8 pieces of 4 k);
  // stored along the output index: piece q = t + 64 h is k-row q / 16,
  // outputs 4 (q % 16) .. + 3
  auto load = [&](int k0) {
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const int q = tid + 64 * h;
      ra[h] = J.ta ? *reinterpret_cast<const float4*>(J.A + (int64_t)(k0 + (q >> 4)) * d + i0 + 4 * (q & 15))
                   : *reinterpret_cast<const float4*>(J.A + (int64_t)(i0 + tid) * d + k0 + 4 * h);
      rb[h] = J.tb ? *reinterpret_cast<const float4*>(J.B + (int64_t)(j0 + tid) * d + k0 + 4 * h)
                   : *reinterpret_cast<const float4*>(J.B + (int64_t)(k0 + (q >> 4)) * d + j0 + 4 * (q & 15));
    }
  };
  auto store = [&]() {
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const int q = tid + 64 * h;
      if (J.ta) {
        *reinterpret_cast<float4*>(&As[q >> 4][4 * (q & 15)]) = ra[h];
      } else {
        As[4 * h][tid] = ra[h].x;
        As[4 * h + 1][tid] = ra[h].y;
        As[4 * h + 2][tid] = ra[h].z;
        As[4 * h + 3][tid] = ra[h].w;
      }
      if (J.tb) {
        Bs[4 * h][tid] = rb[h].x;
        Bs[4 * h + 1][tid] = rb[h].y;
        Bs[4 * h + 2][tid] = rb[h].z;
        Bs[4 * h + 3][tid] = rb[h].w;
      } else {
        *reinterpret_cast<float4*>(&Bs[q >> 4][4 * (q & 15)]) = rb[h];
      }
    }
  };
  // acc[r][p]: row r (0-3: 4 ty + r, 4-7: 32 + 4 ty + r - 4), column pair p
  // (0, 1: 4 tx + {0, 1}, {2, 3}; 2, 3: 32 + 4 tx + ...)
  uint64_t acc[8][4];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0ull;
  load(l0);
  for (int k0 = l0; k0 < l0 + part; k0 += 32) {
    __syncthreads();
    store();
    __syncthreads();
    if (k0 + 32 < l0 + part) load(k0 + 32);
#pragma unroll
    for (int kk = 0; kk < 32; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][4 * ty]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][32 + 4 * ty]);
      const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(&Bs[kk][4 * tx]);
      const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(&Bs[kk][32 + 4 * tx]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const uint64_t aa = pack_f2(av[r], av[r]);
        ffma2(acc[r][0], b0.x, aa);
        ffma2(acc[r][1], b0.y, aa);
        ffma2(acc[r][2], b1.x, aa);
        ffma2(acc[r][3], b1.y, aa);
      }
    }
  }
  // this thread's outputs as rows of two float4 (columns 4 tx.., 32 + 4 tx..)
  auto row_of = [&](int r) { return r < 4 ? 4 * ty + r : 32 + 4 * ty + r - 4; };
  auto piece = [&](int r, int half) {
    const float2 lo = unpack_f2(acc[r][2 * half]), hi = unpack_f2(acc[r][2 * half + 1]);
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  };
  if constexpr (SPLIT == 1) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float* c = J.C + (int64_t)(i0 + row_of(r)) * d + j0;
      *reinterpret_cast<float4*>(c + 4 * tx) = piece(r, 0);
      *reinterpret_cast<float4*>(c + 32 + 4 * tx) = piece(r, 1);
    }
  } else {
    __shared__ __align__(16) float Ps[64][64];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      *reinterpret_cast<float4*>(&Ps[row_of(r)][4 * tx]) = piece(r, 0);
      *reinterpret_cast<float4*>(&Ps[row_of(r)][32 + 4 * tx]) = piece(r, 1);
    }
    cluster_sync();              // every partial tile of the cluster written
    constexpr int kRows = 64 / SPLIT;
    const uint32_t rank = cluster_ctarank();
    for (int e = tid; e < kRows * 16; e += 64) {
      const int row = (int)rank * kRows + e / 16, c4 = e % 16;
      const uint32_t local = smem_u32(&Ps[row][4 * c4]);
      float4 v = ld_dsmem_f4(mapa_shared(local, 0));
#pragma unroll
      for (int q = 1; q < SPLIT; ++q) {
        const float4 w = ld_dsmem_f4(mapa_shared(local, (uint32_t)q));
        v.x += w.x;
        v.y += w.y;
        v.z += w.z;
        v.w += w.w;
      }
      *reinterpret_cast<float4*>(J.C + (int64_t)(i0 + row) * d + j0 + 4 * c4) = v;
    }
    cluster_sync();              // peers done reading this CTA's tile
  }
}

constexpr int kDdSplit = 4;

// The products of one batch (its first `jobs` entries) on stream s: split
// over clusters when d is a multiple of 32 kDdSplit, one block per tile when
// d is a multiple of 64, else the general kernel.
sf_status launch_dd(const DdBatch& bt, int jobs, cudaStream_t s) {
  const int d = bt.d;
  const unsigned tiles = (unsigned)ceil_div(d, 64);
  if (d % (32 * kDdSplit) == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * kDdSplit, tiles, (unsigned)jobs);
    cfg.blockDim = dim3(64);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kDdSplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    SF_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_gemm_dd64<kDdSplit>, bt), "launch k_gemm_dd64");
  } else if (d % 64 == 0) {
    k_gemm_dd64<1><<<dim3(tiles, tiles, (unsigned)jobs), 64, 0, s>>>(bt);
  } else {
    k_gemm_dd<<<dim3(tiles, tiles, (unsigned)jobs), 256, 0, s>>>(bt);
  }
  return check_launch("k_gemm_dd");
}

// H_P = 2 S - X (= S + C with C = S - X, X = A_P S A_Q), H_Q = H_P^T, and
// this block's partial sums of S * S and W1 * W2 (W1 = S A_Q, W2 = A_P S).
__global__ void __launch_bounds__(256) k_fit_combine(const float* __restrict__ S, const float* __restrict__ X,
                                                     const float* __restrict__ W1, const float* __restrict__ W2,
                                                     int d, float* __restrict__ HP, float* __restrict__ HQ,
                                                     double* __restrict__ part) {
  __shared__ float red[2][8];
  const int64_t dd = (int64_t)d * d;
  float s2 = 0.0f, ww = 0.0f;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < dd; t += (int64_t)gridDim.x * blockDim.x) {
    const float s = S[t];
    const float h = 2.0f * s - X[t];
    HP[t] = h;
    HQ[(t % d) * d + t / d] = h;
    s2 = fmaf(s, s, s2);
    ww = fmaf(W1[t], W2[t], ww);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    ww += __shfl_xor_sync(0xffffffffu, ww, o);
  }
  if (lane == 0) {
    red[0][warp] = s2;
    red[1][warp] = ww;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.0f, b = 0.0f;
    for (int w = 0; w < 8; ++w) {
      a += red[0][w];
      b += red[1][w];
    }
    part[2 * blockIdx.x] = (double)a;
    part[2 * blockIdx.x + 1] = (double)b;
  }
}

// g[r k + s] = -2 (<X[r, :], H[c_s, :]> - sum_t v_t K[c_t][c_s]) for the k
// stored entries (c_t, v_t) of row r; one warp per row, the lanes along d.
// For k <= 8 the k dot products share each load of X[r, :] and are summed
// side by side; every sum has a fixed lane order and a fixed butterfly.
__global__ void __launch_bounds__(256) k_fit_rowgrad(const float* __restrict__ X, int64_t rows, int d,
                                                     const int32_t* __restrict__ idx, const float* __restrict__ val,
                                                     int k, const float* __restrict__ H, const float* __restrict__ K,
                                                     float* __restrict__ g) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const float* x = X + r * d;
  const int32_t* ir = idx + r * k;
  const float* vr = val + r * k;
  if (k <= 8) {
    int c[8];
    float p[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      c[s] = s < k ? ir[s] : 0;
      p[s] = 0.0f;
    }
    for (int u = lane; u < d; u += 32) {
      const float xu = x[u];
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (s < k) p[s] = fmaf(xu, H[(int64_t)c[s] * d + u], p[s]);
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (s >= k) break;
      float kt = 0.0f;
      if (lane < k) kt = vr[lane] * K[(int64_t)ir[lane] * d + c[s]];
      float ps = p[s];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        ps += __shfl_xor_sync(0xffffffffu, ps, o);
        kt += __shfl_xor_sync(0xffffffffu, kt, o);
      }
      if (lane == 0) g[r * k + s] = -2.0f * (ps - kt);
    }
    return;
  }
  for (int s = 0; s < k; ++s) {
    const int c = ir[s];
    const float* h = H + (int64_t)c * d;
    float p = 0.0f;
    for (int u = lane; u < d; u += 32) p = fmaf(x[u], h[u], p);
    float kt = 0.0f;
    for (int t = lane; t < k; t += 32) kt = fmaf(vr[t], K[(int64_t)ir[t] * d + c], kt);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      p += __shfl_xor_sync(0xffffffffu, p, o);
      kt += __shfl_xor_sync(0xffffffffu, kt, o);
    }
    if (lane == 0) g[r * k + s] = -2.0f * (p - kt);
  }
}

// The same gradients when d is a multiple of 128 and k <= 8, with the lanes
// along d in 16-byte pieces: each lane reads 4 consecutive elements of X[r]
// and of the k rows of H per step, all nine loads issued before the
// multiply-adds, so a warp has d / 128 steps of loads in flight instead of
// d / 32.  Each lane sums its pieces in order; the lanes combine in a fixed
// butterfly.
__global__ void __launch_bounds__(256) k_fit_rowgrad4(const float* __restrict__ X, int64_t rows, int d,
                                                      const int32_t* __restrict__ idx, const float* __restrict__ val,
                                                      int k, const float* __restrict__ H, const float* __restrict__ K,
                                                      float* __restrict__ g) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const float* x = X + r * d;
  const int32_t* ir = idx + r * k;
  const float* vr = val + r * k;
  const float* h[8];
  float p[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    h[s] = H + (int64_t)(s < k ? ir[s] : ir[0]) * d;
    p[s] = 0.0f;
  }
  for (int u = 4 * lane; u < d; u += 128) {
    const float4 xu = *reinterpret_cast<const float4*>(x + u);
    float4 hu[8];
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s < k) hu[s] = *reinterpret_cast<const float4*>(h[s] + u);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (s < k) {
        p[s] = fmaf(xu.x, hu[s].x, p[s]);
        p[s] = fmaf(xu.y, hu[s].y, p[s]);
        p[s] = fmaf(xu.z, hu[s].z, p[s]);
        p[s] = fmaf(xu.w, hu[s].w, p[s]);
      }
    }
  }
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    if (s >= k) break;
    float kt = 0.0f;
    if (lane < k) kt = vr[lane] * K[(int64_t)ir[lane] * d + ir[s]];
    float ps = p[s];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ps += __shfl_xor_sync(0xffffffffu, ps, o);
      kt += __shfl_xor_sync(0xffffffffu, kt, o);
    }
    if (lane == 0) g[r * k + s] = -2.0f * (ps - kt);
  }
}

// L = sum(G^2) - 2 sum(S^2) + sum(W1 W2), from the block partials, in fp64
// and in a fixed order.
__global__ void __launch_bounds__(1024) k_fit_loss(const double* __restrict__ g2, int64_t n_g2,
                                                   const double* __restrict__ part, int n_part,
                                                   double* __restrict__ loss) {
  __shared__ double red[3][1024];
  double a = 0.0, b = 0.0, c = 0.0;
  for (int64_t i = threadIdx.x; i < n_g2; i += blockDim.x) a += g2[i];
  for (int i = threadIdx.x; i < n_part; i += blockDim.x) {
    b += part[2 * i];
    c += part[2 * i + 1];
  }
  red[0][threadIdx.x] = a;
  red[1][threadIdx.x] = b;
  red[2][threadIdx.x] = c;
  __syncthreads();
  for (int st = blockDim.x / 2; st > 0; st >>= 1) {
    if ((int)threadIdx.x < st)
      for (int q = 0; q < 3; ++q) red[q][threadIdx.x] += red[q][threadIdx.x + st];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = red[0][0] - 2.0 * red[1][0] + red[2][0];
}

// val <- val - lr * g for every stored entry, written to the ELL copy, the
// CSC values and the window-major list.
__global__ void k_fit_update(int64_t nnz, float lr, const float* __restrict__ g, float* __restrict__ ell_val,
                             float* __restrict__ csc_val, int2* __restrict__ went, const int32_t* __restrict__ e2c,
                             const int32_t* __restrict__ e2w) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += (int64_t)gridDim.x * blockDim.x) {
    const float v = fmaf(-lr, g[e], ell_val[e]);
    ell_val[e] = v;
    const int32_t c = e2c[e], w = e2w[e];
    if (c >= 0) csc_val[c] = v;
    if (w >= 0) went[w].y = __float_as_int(v);
  }
}

constexpr int kCombineBlocks = 128;

struct FitPlan {
  CompressPlan cp;
  GatherPlan gt;
  size_t off_gt, off_t, off_tp, off_dd, off_gp, off_gq, off_g2, off_part, bytes;
  int64_t n_g2;
};

FitPlan plan_fit(int64_t m, int64_t n, int d, size_t es, int kP, int kQ) {
  FitPlan f;
  f.cp = plan_compress(m, n, d);
  f.gt = plan_gather(n, m, d);
  size_t off = f.cp.bytes;
  f.off_gt = off;
  off = align_up(off + (size_t)m * n * es, 256);
  f.off_t = off;
  off = align_up(off + (size_t)m * d * 4, 256);
  f.off_tp = off;
  off += f.gt.partial_bytes;
  f.off_dd = off;
  off = align_up(off + (size_t)10 * d * d * 4, 256);
  f.off_gp = off;
  off = align_up(off + (size_t)m * kP * 4, 256);
  f.off_gq = off;
  off = align_up(off + (size_t)n * kQ * 4, 256);
  f.n_g2 = ceil_div<int64_t>(m, 64) * ceil_div<int64_t>(n, 64);
  f.off_g2 = off;
  off = align_up(off + (size_t)f.n_g2 * 8, 256);
  f.off_part = off;
  off = align_up(off + (size_t)kCombineBlocks * 2 * 8, 256);
  f.bytes = off;
  return f;
}

}  // namespace
}  // namespace sf

extern "C" {

size_t lsp_fit_workspace_bytes(int64_t m, int64_t n, int32_t d, sf_dtype g_dtype) {
  if (m < 1 || n < 1 || d < 1) return 0;
  // the k of the projectors only sizes the internal gradient buffers: take the largest k accepted
  return sf::plan_fit(m, n, d, g_dtype == SF_BF16 ? 2 : 4, 64, 64).bytes;
}

sf_status lsp_projector_fit_step(lsp_projector P, lsp_projector Q, const void* G, sf_dtype g_dtype, int64_t m,
                                 int64_t n, double lr, double* loss, float* grad_P, float* grad_Q, void* ws,
                                 size_t ws_bytes, void* stream_) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("lsp_projector_fit_step");
  SF_TRY(sf::check_proj(P, "P"));
  SF_TRY(sf::check_proj(Q, "Q"));
  if (P == Q) return fail(SF_ERR_INVALID, "P and Q must be different projector handles");
  if (P->bad_ids || Q->bad_ids)
    return fail(SF_ERR_INVALID, "a projector had column ids outside [0, d) at creation; its values cannot be fitted");
  if (!G) return fail(SF_ERR_INVALID, "G is NULL");
  if (P->rows != m || Q->rows != n)
    return fail(SF_ERR_INVALID, "P has %lld rows, Q %lld: need m = %lld, n = %lld", (long long)P->rows,
                (long long)Q->rows, (long long)m, (long long)n);
  if (P->d != Q->d) return fail(SF_ERR_INVALID, "P and Q differ in d (%d vs %d)", P->d, Q->d);
  if (g_dtype != SF_BF16 && g_dtype != SF_FP32) return fail(SF_ERR_INVALID, "g_dtype must be SF_BF16 or SF_FP32");
  if (!(lr == lr) || lr > 3.0e38 || lr < -3.0e38) return fail(SF_ERR_INVALID, "lr must be finite");
  const int d = P->d;
  const size_t es = g_dtype == SF_BF16 ? 2 : 4;
  const sf::FitPlan f = sf::plan_fit(m, n, d, es, 64, 64);
  if (!ws || ws_bytes < f.bytes || (reinterpret_cast<uintptr_t>(ws) % 256) != 0)
    return fail(SF_ERR_INVALID, "workspace needs %zu bytes, 256-byte aligned (got %zu)", f.bytes, ws_bytes);
  cudaStream_t s = sf::as_stream(stream_);
  char* w = static_cast<char*>(ws);
  float* U = reinterpret_cast<float*>(w + f.cp.off_rt);
  float* Ut = reinterpret_cast<float*>(w + f.cp.off_rtp);
  float* Sp = reinterpret_cast<float*>(w + f.cp.off_sp);
  void* Gt = w + f.off_gt;
  float* T = reinterpret_cast<float*>(w + f.off_t);
  float* Tp = reinterpret_cast<float*>(w + f.off_tp);
  float* dd = reinterpret_cast<float*>(w + f.off_dd);
  const size_t dd1 = (size_t)d * d;
  float *S = dd, *AP = dd + dd1, *AQ = dd + 2 * dd1, *W1 = dd + 3 * dd1, *W2 = dd + 4 * dd1, *X = dd + 5 * dd1,
        *K1 = dd + 6 * dd1, *K2 = dd + 7 * dd1, *HP = dd + 8 * dd1, *HQ = dd + 9 * dd1;
  float* gP = grad_P ? grad_P : reinterpret_cast<float*>(w + f.off_gp);
  float* gQ = grad_Q ? grad_Q : reinterpret_cast<float*>(w + f.off_gq);
  double* g2 = reinterpret_cast<double*>(w + f.off_g2);
  double* part = reinterpret_cast<double*>(w + f.off_part);

  // U = G^T P and S = P^T G Q (the compress pair); G^T with the sum of G^2; T = G Q
  const dim3 tgrid((unsigned)ceil_div<int64_t>(n, 64), (unsigned)ceil_div<int64_t>(m, 64));
  if (tgrid.y > 65535u) return fail(SF_ERR_UNSUPPORTED, "m = %lld is too large for the fit step", (long long)m);
  if (g_dtype == SF_FP32) {
    const float* Gf = static_cast<const float*>(G);
    SF_TRY(sf::launch_gather<float>(P, Gf, n, n, f.cp.g1, U, Ut, s));
    sf::k_transpose_sumsq<float><<<tgrid, 256, 0, s>>>(Gf, m, n, static_cast<float*>(Gt), g2);
    SF_TRY(sf::check_launch("k_transpose_sumsq"));
    SF_TRY(sf::launch_gather<float>(Q, static_cast<const float*>(Gt), m, m, f.gt, T, Tp, s));
  } else {
    const __nv_bfloat16* Gb = static_cast<const __nv_bfloat16*>(G);
    SF_TRY(sf::launch_gather<__nv_bfloat16>(P, Gb, n, n, f.cp.g1, U, Ut, s));
    sf::k_transpose_sumsq<__nv_bfloat16><<<tgrid, 256, 0, s>>>(Gb, m, n, static_cast<__nv_bfloat16*>(Gt), g2);
    SF_TRY(sf::check_launch("k_transpose_sumsq"));
    SF_TRY(sf::launch_gather<__nv_bfloat16>(Q, static_cast<const __nv_bfloat16*>(Gt), m, m, f.gt, T, Tp, s));
  }
  SF_TRY(sf::launch_stage2(Q, U, d, d, f.cp.g2, S, Sp, s));

  // Gram matrices A_P = P^T P, A_Q = Q^T Q from the sparse forms, then the
  // five d x d products
  const size_t gram_smem = (size_t)sf::kGramWarps * d * 4;
  SF_TRY(sf::allow_dynamic_smem(reinterpret_cast<const void*>(&sf::k_gram_sparse), gram_smem));
  const unsigned gram_grid = (unsigned)ceil_div(d, sf::kGramWarps / sf::kGramSplit);
  sf::k_gram_sparse<<<gram_grid, 32 * sf::kGramWarps, gram_smem, s>>>(P->col_ptr, P->row_idx, P->csc_val,
                                                                       P->ell_idx, P->ell_val, P->k, d, AP);
  SF_TRY(sf::check_launch("k_gram_sparse"));
  sf::k_gram_sparse<<<gram_grid, 32 * sf::kGramWarps, gram_smem, s>>>(Q->col_ptr, Q->row_idx, Q->csc_val,
                                                                       Q->ell_idx, Q->ell_val, Q->k, d, AQ);
  SF_TRY(sf::check_launch("k_gram_sparse"));
  sf::DdBatch b1{};
  b1.d = d;
  b1.job[0] = {S, AQ, W1, 0, 0};   // W1 = S A_Q
  b1.job[1] = {AP, S, W2, 0, 0};   // W2 = A_P S
  SF_TRY(sf::launch_dd(b1, 2, s));
  sf::DdBatch b2{};
  b2.d = d;
  b2.job[0] = {W2, AQ, X, 0, 0};   // X = A_P S A_Q
  b2.job[1] = {W1, S, K1, 0, 1};   // K1 = S A_Q S^T
  b2.job[2] = {S, W2, K2, 1, 0};   // K2 = S^T A_P S
  SF_TRY(sf::launch_dd(b2, 3, s));
  sf::k_fit_combine<<<sf::kCombineBlocks, 256, 0, s>>>(S, X, W1, W2, d, HP, HQ, part);
  SF_TRY(sf::check_launch("k_fit_combine"));

  // gradients at the stored positions, the loss, then the step
  auto rowgrad = [&](const float* X, int64_t rows, const lsp_projector_s* A, const float* H, const float* K,
                     float* g) {
    const unsigned grid = (unsigned)ceil_div<int64_t>(rows, 8);
    if (d % 128 == 0 && A->k <= 8 && reinterpret_cast<uintptr_t>(X) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(H) % 16 == 0)
      sf::k_fit_rowgrad4<<<grid, 256, 0, s>>>(X, rows, d, A->ell_idx, A->ell_val, A->k, H, K, g);
    else
      sf::k_fit_rowgrad<<<grid, 256, 0, s>>>(X, rows, d, A->ell_idx, A->ell_val, A->k, H, K, g);
  };
  rowgrad(T, m, P, HP, K1, gP);
  rowgrad(U, n, Q, HQ, K2, gQ);
  SF_TRY(sf::check_launch("k_fit_rowgrad"));
  if (loss) {
    sf::k_fit_loss<<<1, 1024, 0, s>>>(g2, f.n_g2, part, sf::kCombineBlocks, loss);
    SF_TRY(sf::check_launch("k_fit_loss"));
  }
  const float lr32 = (float)lr;
  if (lr32 != 0.0f) {
    const int nsm = sf::sm_count();
    const int64_t nP = P->rows * (int64_t)P->k, nQ = Q->rows * (int64_t)Q->k;
    sf::k_fit_update<<<(unsigned)std::min<int64_t>(ceil_div<int64_t>(nP, 256), nsm * 8), 256, 0, s>>>(
        nP, lr32, gP, P->ell_val, P->csc_val, P->went, P->ell2csc, P->ell2went);
    sf::k_fit_update<<<(unsigned)std::min<int64_t>(ceil_div<int64_t>(nQ, 256), nsm * 8), 256, 0, s>>>(
        nQ, lr32, gQ, Q->ell_val, Q->csc_val, Q->went, Q->ell2csc, Q->ell2went);
    SF_TRY(sf::check_launch("k_fit_update"));
  }
  return SF_OK;
}

sf_status lsp_projector_export_values(lsp_projector p, float* val, void* stream_) {
  sf::clear_error();
  SF_TRY(sf::check_proj(p, "p"));
  if (!val) return fail(SF_ERR_INVALID, "val is NULL");
  SF_CUDA_TRY(cudaMemcpyAsync(val, p->ell_val, (size_t)p->rows * p->k * 4, cudaMemcpyDeviceToDevice,
                              sf::as_stream(stream_)),
              "export values");
  return SF_OK;
}

}  // extern "C"

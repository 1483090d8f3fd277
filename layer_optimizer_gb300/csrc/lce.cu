// Fused linear cross-entropy: loss and gradients of the softmax
// cross-entropy of a linear output layer, chunked over tokens so that the
// full logits tensor is never held.
//
// SlideFormer ("An Efficient Heterogeneous Co-Design for Fine-Tuning on a
// Single GPU"; the summaries' kernel lists, "Fused LinearCrossEntropy")
// fuses the output projection with the loss and computes the gradients in
// small blocks, so the logits (tokens x vocabulary, larger than every other
// activation for big vocabularies) never exist in full.  For each chunk of
// tokens c:
//   Z_c  = H_c W^T                      tensor cores, fp32 [chunk][V]
//   lse  = logsumexp over each row of Z_c, from (max, sum exp) pairs the
//          logits GEMM's epilogue writes per row and 256-column tile, and
//          the rows' losses
//   G_c  = (softmax(Z_c) - onehot(y_c)) / n  rounded to bf16, written both
//          as [chunk][V] and transposed [V][chunk]
//   dH_c = G_c W                        tensor cores (W^T made once per call)
//   dW  += G_c^T H_c                    tensor cores (H_c^T made per chunk)
// n is the number of tokens whose label is not ignore_index.  The three
// products run on the tensor-core GEMM (tc_gemm.cu); the row statistics and
// the gradient tile are fp32 CUDA-core kernels.  Memory: one chunk of
// logits (fp32) and two of the bf16 gradient instead of N x V.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.h"
#include "ptx.cuh"

namespace sf {
namespace {

// out[c][r] = in[r][c] for a rows x cols bf16 matrix (row pitches ld_in,
// ld_out; cols, ld_in and ld_out even), through a padded 64 x 64 tile held as
// 32-bit words: coalesced 4-byte loads of column pairs, and each output word
// (rows 2p and 2p + 1 of one column) assembled from two tile words.
__global__ void __launch_bounds__(256) k_transpose_bf16(const uint16_t* __restrict__ in, int64_t rows,
                                                        int64_t cols, int64_t ld_in, uint16_t* __restrict__ out,
                                                        int64_t ld_out) {
  __shared__ uint32_t tile[64][33];
  const int64_t r0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int q = threadIdx.x + 256 * k;       // 64 rows x 32 words
    const int r = q >> 5, w = q & 31;
    const int64_t i = r0 + r, j = c0 + 2 * w;
    uint32_t v = 0;
    if (i < rows && j < cols) v = *reinterpret_cast<const uint32_t*>(in + i * ld_in + j);
    tile[r][w] = v;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int q = threadIdx.x + 256 * k;       // 64 output rows (columns c) x 32 words (row pairs p)
    const int c = q >> 5, p = q & 31;
    const int64_t j = c0 + c, i = r0 + 2 * p;
    if (j < cols && i < rows) {
      const uint32_t lo = tile[2 * p][c >> 1], hi = tile[2 * p + 1][c >> 1];
      // the half of each word that holds column c (low half = even column)
      const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
      *reinterpret_cast<uint32_t*>(out + j * ld_out + i) = __byte_perm(lo, hi, sel);
    }
  }
}

// Number n of labelled tokens (label != ignore and in [0, V)); a label that
// is neither is counted as unlabelled and flagged.  inv_n = 1/n (0 if n = 0).
__global__ void __launch_bounds__(1024) k_lce_count(const int32_t* __restrict__ labels, int64_t N, int64_t V,
                                                    int32_t ignore, int64_t* __restrict__ n_out,
                                                    float* __restrict__ inv_n) {
  __shared__ int64_t red[1024];
  int64_t c = 0;
  bool bad = false;
  for (int64_t i = threadIdx.x; i < N; i += blockDim.x) {
    const int32_t y = labels[i];
    if (y == ignore) continue;
    if (y < 0 || y >= V) bad = true;
    else ++c;
  }
  if (bad) atomicOr(&g_device_error, kDevErrIndex);
  red[threadIdx.x] = c;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *n_out = red[0];
    *inv_n = red[0] > 0 ? (float)(1.0 / (double)red[0]) : 0.0f;
  }
}

__device__ __forceinline__ bool labelled(int32_t y, int32_t ignore, int64_t V) {
  return y != ignore && y >= 0 && y < V;
}

// (m, s) pairs meaning "s = sum of exp(x - m)" combined into one.
__device__ __forceinline__ void combine_stats(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float mn = fmaxf(m, m2);
  s = s * expf(m - mn) + s2 * expf(m2 - mn);
  m = mn;
}

// One warp per row of the chunk: lse = log sum_j exp(z_j) from the logits
// GEMM's per-tile (max, sum of exp) pairs, combined in a fixed order (lanes
// over tiles, then a butterfly); the row's loss lse - z[y] (0 for an
// unlabelled token).
__global__ void __launch_bounds__(256) k_lce_lse(const float2* __restrict__ stats, int n_tiles, int64_t rows,
                                                 const float* __restrict__ Z, int64_t V,
                                                 const int32_t* __restrict__ labels, int32_t ignore,
                                                 float* __restrict__ lse, float* __restrict__ row_loss) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  float m = -INFINITY, s = 0.0f;
  for (int t = lane; t < n_tiles; t += 32) {
    const float2 p = stats[r * n_tiles + t];
    combine_stats(m, s, p.x, p.y);
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    // the same pair order on both lanes of the exchange: lower lane first
    if (lane & o) {
      float mm = m2, ss = s2;
      combine_stats(mm, ss, m, s);
      m = mm;
      s = ss;
    } else {
      combine_stats(m, s, m2, s2);
    }
  }
  if (lane == 0) {
    const float l = m + logf(s);
    lse[r] = l;
    const int32_t y = labels[r];
    row_loss[r] = labelled(y, ignore, V) ? l - Z[r * V + y] : 0.0f;
  }
}

// The gradient tile: g = (exp(z - lse) - [j == y]) * inv_n (0 for an
// unlabelled row), rounded to bf16, written to G [rows][V] and Gt
// [V][ld_gt] (columns = rows of the chunk).  Each thread takes column pairs
// (8-byte loads of Z, 4-byte stores of G); the transposed copy goes through
// a padded tile of 32-bit words like k_transpose_bf16.  V, ld_gt even.
__global__ void __launch_bounds__(256) k_lce_grad(const float* __restrict__ Z, int64_t rows, int64_t V,
                                                  const float* __restrict__ lse, const int32_t* __restrict__ labels,
                                                  int32_t ignore, const float* __restrict__ inv_n,
                                                  __nv_bfloat16* __restrict__ G, __nv_bfloat16* __restrict__ Gt,
                                                  int64_t ld_gt) {
  __shared__ uint32_t tile[64][33];
  const int64_t r0 = (int64_t)blockIdx.y * 64, j0 = (int64_t)blockIdx.x * 64;
  const float sc = *inv_n;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int q = threadIdx.x + 256 * k;       // 64 rows x 32 column pairs
    const int r = q >> 5, w = q & 31;
    const int64_t i = r0 + r, j = j0 + 2 * w;
    uint32_t word = 0;
    if (i < rows && j < V) {
      const int32_t y = labels[i];
      float g0 = 0.0f, g1 = 0.0f;
      if (labelled(y, ignore, V)) {
        const float2 z = *reinterpret_cast<const float2*>(Z + i * V + j);
        const float l = lse[i];
        g0 = (expf(z.x - l) - (j == y ? 1.0f : 0.0f)) * sc;
        g1 = (expf(z.y - l) - (j + 1 == y ? 1.0f : 0.0f)) * sc;
      }
      const __nv_bfloat162 h = __floats2bfloat162_rn(g0, g1);
      word = *reinterpret_cast<const uint32_t*>(&h);
      *reinterpret_cast<uint32_t*>(G + i * V + j) = word;
    }
    tile[r][w] = word;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int q = threadIdx.x + 256 * k;       // 64 columns c x 32 row pairs p
    const int c = q >> 5, p = q & 31;
    const int64_t j = j0 + c, i = r0 + 2 * p;
    if (j < V && i < rows) {
      const uint32_t lo = tile[2 * p][c >> 1], hi = tile[2 * p + 1][c >> 1];
      const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
      *reinterpret_cast<uint32_t*>(Gt + j * ld_gt + i) = __byte_perm(lo, hi, sel);
    }
  }
}

// loss = sum of the rows' losses * inv_n, in fp64 and a fixed order.
__global__ void __launch_bounds__(1024) k_lce_loss(const float* __restrict__ row_loss, int64_t N,
                                                   const float* __restrict__ inv_n, double* __restrict__ loss) {
  __shared__ double red[1024];
  double a = 0.0;
  for (int64_t i = threadIdx.x; i < N; i += blockDim.x) a += (double)row_loss[i];
  red[threadIdx.x] = a;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = red[0] * (double)*inv_n;
}

struct LcePlan {
  size_t off_z, off_g, off_gt, off_wt, off_ht, off_lse, off_rowloss, off_n, off_stats, bytes;
};

LcePlan plan_lce(int64_t N, int64_t D, int64_t V, int64_t chunk) {
  LcePlan p;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = (off + bytes + 255) / 256 * 256;
    return o;
  };
  p.off_z = take((size_t)chunk * V * 4);
  p.off_g = take((size_t)chunk * V * 2);
  p.off_gt = take((size_t)V * chunk * 2);
  p.off_wt = take((size_t)D * V * 2);
  p.off_ht = take((size_t)D * chunk * 2);
  p.off_lse = take((size_t)chunk * 4);
  p.off_rowloss = take((size_t)N * 4);
  p.off_n = take(16);
  p.off_stats = take((size_t)chunk * ((V + kTcTileN - 1) / kTcTileN) * 8);
  p.bytes = off;
  return p;
}

}  // namespace

int read_and_clear_device_error_lce() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof z);
  return v;
}

}  // namespace sf

extern "C" {

size_t lce_workspace_bytes(int64_t n_tokens, int64_t d, int64_t vocab, int64_t chunk) {
  if (n_tokens < 1 || d < 1 || vocab < 1 || chunk < 1) return 0;
  return sf::plan_lce(n_tokens, d, vocab, std::min(chunk, (n_tokens + 7) / 8 * 8)).bytes;
}

sf_status lce_forward_backward(const void* H, const void* W, const int32_t* labels, int64_t N, int64_t D, int64_t V,
                               int64_t chunk, int32_t ignore_index, double* loss, float* dH, float* dW, void* ws,
                               size_t ws_bytes, void* stream_) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("lce_forward_backward");
  if (!H || !W || !labels) return sf::fail(SF_ERR_INVALID, "H, W or labels is NULL");
  if (N < 1 || D < 1 || V < 1) return sf::fail(SF_ERR_INVALID, "N, D, V must be >= 1");
  if (D % 8 || V % 8) return sf::fail(SF_ERR_UNSUPPORTED, "D and V must be multiples of 8 (16-byte rows)");
  if (chunk < 8 || chunk % 8) return sf::fail(SF_ERR_INVALID, "chunk must be a positive multiple of 8");
  if ((reinterpret_cast<uintptr_t>(H) % 16) || (reinterpret_cast<uintptr_t>(W) % 16))
    return sf::fail(SF_ERR_UNSUPPORTED, "H and W need 16-byte aligned bases");
  if ((dH && reinterpret_cast<uintptr_t>(dH) % 16) || (dW && reinterpret_cast<uintptr_t>(dW) % 16))
    return sf::fail(SF_ERR_UNSUPPORTED, "dH and dW need 16-byte aligned bases");
  chunk = std::min(chunk, (N + 7) / 8 * 8);
  if ((chunk + 63) / 64 > 65535 || (V + 63) / 64 > (int64_t)INT32_MAX || N > (int64_t)INT32_MAX)
    return sf::fail(SF_ERR_UNSUPPORTED, "sizes too large");
  const sf::LcePlan p = sf::plan_lce(N, D, V, chunk);
  if (!ws || ws_bytes < p.bytes || (reinterpret_cast<uintptr_t>(ws) % 256))
    return sf::fail(SF_ERR_INVALID, "workspace needs %zu bytes, 256-byte aligned (got %zu)", p.bytes, ws_bytes);
  cudaStream_t s = sf::as_stream(stream_);
  char* w = static_cast<char*>(ws);
  float* Z = reinterpret_cast<float*>(w + p.off_z);
  __nv_bfloat16* G = reinterpret_cast<__nv_bfloat16*>(w + p.off_g);
  __nv_bfloat16* Gt = reinterpret_cast<__nv_bfloat16*>(w + p.off_gt);
  uint16_t* Wt = reinterpret_cast<uint16_t*>(w + p.off_wt);
  uint16_t* Ht = reinterpret_cast<uint16_t*>(w + p.off_ht);
  float* lse = reinterpret_cast<float*>(w + p.off_lse);
  float* row_loss = reinterpret_cast<float*>(w + p.off_rowloss);
  int64_t* n_valid = reinterpret_cast<int64_t*>(w + p.off_n);
  float* inv_n = reinterpret_cast<float*>(w + p.off_n + 8);
  float2* stats = reinterpret_cast<float2*>(w + p.off_stats);
  const int n_vt = (int)((V + sf::kTcTileN - 1) / sf::kTcTileN);
  const uint16_t* Hb = static_cast<const uint16_t*>(H);
  const bool grads = dH || dW;

  sf::k_lce_count<<<1, 1024, 0, s>>>(labels, N, V, ignore_index, n_valid, inv_n);
  SF_TRY(sf::check_launch("k_lce_count"));
  if (dH) {
    sf::k_transpose_bf16<<<dim3((unsigned)sf::ceil_div<int64_t>(D, 64), (unsigned)sf::ceil_div<int64_t>(V, 64)), 256, 0, s>>>(
        static_cast<const uint16_t*>(W), V, D, D, Wt, V);
    SF_TRY(sf::check_launch("k_transpose_bf16"));
  }
  for (int64_t c0 = 0; c0 < N; c0 += chunk) {
    const int64_t rows = std::min(chunk, N - c0);
    SF_TRY(sf::tc_gemm_abt(Hb + c0 * D, W, Z, rows, V, D, D, D, V, 1.0f, false, s, stats));
    sf::k_lce_lse<<<(unsigned)sf::ceil_div<int64_t>(rows, 8), 256, 0, s>>>(stats, n_vt, rows, Z, V, labels + c0,
                                                                             ignore_index, lse, row_loss + c0);
    SF_TRY(sf::check_launch("k_lce_lse"));
    if (!grads) continue;
    sf::k_lce_grad<<<dim3((unsigned)sf::ceil_div<int64_t>(V, 64), (unsigned)sf::ceil_div<int64_t>(rows, 64)), 256, 0, s>>>(
        Z, rows, V, lse, labels + c0, ignore_index, inv_n, G, Gt, chunk);
    SF_TRY(sf::check_launch("k_lce_grad"));
    if (dH) SF_TRY(sf::tc_gemm_abt(G, Wt, dH + c0 * D, rows, D, V, V, V, D, 1.0f, false, s));
    if (dW) {
      sf::k_transpose_bf16<<<dim3((unsigned)sf::ceil_div<int64_t>(D, 64), (unsigned)sf::ceil_div<int64_t>(rows, 64)), 256, 0,
                             s>>>(Hb + c0 * D, rows, D, D, Ht, chunk);
      SF_TRY(sf::check_launch("k_transpose_bf16"));
      SF_TRY(sf::tc_gemm_abt(Gt, Ht, dW, V, D, rows, chunk, chunk, D, 1.0f, c0 > 0, s));
    }
  }
  if (loss) {
    sf::k_lce_loss<<<1, 1024, 0, s>>>(row_loss, N, inv_n, loss);
    SF_TRY(sf::check_launch("k_lce_loss"));
  }
  return SF_OK;
}

}  // extern "C"

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
//   G_c  = (softmax(Z_c) - onehot(y_c)) / n  rounded to bf16 [chunk][V]
//   dH_c = G_c W                        tensor cores, W read MN-major
//   dW  += G_c^T H_c                    tensor cores, G_c and H_c read MN-major
// n is the number of tokens whose label is not ignore_index.  The three
// products run on the tensor-core GEMM (tc_gemm.cu), which reads either
// layout of an operand, so no transposed copy of W, G or H is made; the row
// statistics and the gradient are fp32 CUDA-core kernels.  Memory: one
// chunk of logits (fp32) and one of the bf16 gradient instead of N x V.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.h"
#include "ptx.cuh"

namespace sf {
namespace {

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

// The gradient: g = (exp(z - lse) - [j == y]) * inv_n (0 for an unlabelled
// row), rounded to bf16, G [rows][V].  A CTA takes 8192 columns of one row:
// each thread 8 float4 loads of Z in flight (read once, streaming) and
// 8-byte stores of 4 bf16.  V is a multiple of 8.
constexpr int kGradCols = 256 * 4 * 8;
__global__ void __launch_bounds__(256) k_lce_grad(const float* __restrict__ Z, int64_t rows, int64_t V,
                                                  const float* __restrict__ lse, const int32_t* __restrict__ labels,
                                                  int32_t ignore, const float* __restrict__ inv_n,
                                                  __nv_bfloat16* __restrict__ G) {
  const float sc = *inv_n;
  const int64_t j0 = (int64_t)blockIdx.x * kGradCols + 4 * threadIdx.x;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    const int32_t y = labels[r];
    const bool on = labelled(y, ignore, V);
    const float l = lse[r];
    const float* zr = Z + r * V;
    __nv_bfloat16* gr = G + r * V;
    float4 z[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t j = j0 + 1024 * u;
      z[u] = (on && j < V) ? __ldcs(reinterpret_cast<const float4*>(zr + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t j = j0 + 1024 * u;
      if (j < V) {
        float g0 = 0.0f, g1 = 0.0f, g2 = 0.0f, g3 = 0.0f;
        if (on) {
          g0 = (expf(z[u].x - l) - (j == y ? 1.0f : 0.0f)) * sc;
          g1 = (expf(z[u].y - l) - (j + 1 == y ? 1.0f : 0.0f)) * sc;
          g2 = (expf(z[u].z - l) - (j + 2 == y ? 1.0f : 0.0f)) * sc;
          g3 = (expf(z[u].w - l) - (j + 3 == y ? 1.0f : 0.0f)) * sc;
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(g0, g1), hi = __floats2bfloat162_rn(g2, g3);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t*>(&lo);
        w.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(gr + j) = w;
      }
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
  size_t off_z, off_g, off_lse, off_rowloss, off_n, off_stats, bytes;
};

// Workspace of one call: the chunk's logits and gradient, its row statistics,
// the row losses of all tokens, the labelled-token count (no dependence on D:
// nothing is transposed).
LcePlan plan_lce(int64_t N, int64_t V, int64_t chunk) {
  LcePlan p;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = (off + bytes + 255) / 256 * 256;
    return o;
  };
  p.off_z = take((size_t)chunk * V * 4);
  p.off_g = take((size_t)chunk * V * 2);
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
  return sf::plan_lce(n_tokens, vocab, std::min(chunk, (n_tokens + 7) / 8 * 8)).bytes;
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
  if (V > (int64_t)INT32_MAX / 2 || N > (int64_t)INT32_MAX || D > (int64_t)INT32_MAX / 2)
    return sf::fail(SF_ERR_UNSUPPORTED, "sizes too large");
  const sf::LcePlan p = sf::plan_lce(N, V, chunk);
  if (!ws || ws_bytes < p.bytes || (reinterpret_cast<uintptr_t>(ws) % 256))
    return sf::fail(SF_ERR_INVALID, "workspace needs %zu bytes, 256-byte aligned (got %zu)", p.bytes, ws_bytes);
  cudaStream_t s = sf::as_stream(stream_);
  char* w = static_cast<char*>(ws);
  float* Z = reinterpret_cast<float*>(w + p.off_z);
  __nv_bfloat16* G = reinterpret_cast<__nv_bfloat16*>(w + p.off_g);
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
  for (int64_t c0 = 0; c0 < N; c0 += chunk) {
    const int64_t rows = std::min(chunk, N - c0);
    SF_TRY(sf::tc_gemm(Hb + c0 * D, false, W, false, Z, rows, V, D, D, D, V, 1.0f, false, s, stats));
    sf::k_lce_lse<<<(unsigned)sf::ceil_div<int64_t>(rows, 8), 256, 0, s>>>(stats, n_vt, rows, Z, V, labels + c0,
                                                                             ignore_index, lse, row_loss + c0);
    SF_TRY(sf::check_launch("k_lce_lse"));
    if (!grads) continue;
    const dim3 grid((unsigned)sf::ceil_div<int64_t>(V, sf::kGradCols), (unsigned)std::min<int64_t>(rows, 65535));
    sf::k_lce_grad<<<grid, 256, 0, s>>>(Z, rows, V, lse, labels + c0, ignore_index, inv_n, G);
    SF_TRY(sf::check_launch("k_lce_grad"));
    // dH_c = G_c W: G_c K-major [rows][V]; W is [V][D] = B stored [K][N]
    if (dH) SF_TRY(sf::tc_gemm(G, false, W, true, dH + c0 * D, rows, D, V, V, D, D, 1.0f, false, s));
    // dW += G_c^T H_c: A = G_c^T stored [K = rows][M = V], B = H_c^T stored [K][N = D]
    if (dW) SF_TRY(sf::tc_gemm(G, true, Hb + c0 * D, true, dW, V, D, rows, V, D, D, 1.0f, c0 > 0, s));
  }
  if (loss) {
    sf::k_lce_loss<<<1, 1024, 0, s>>>(row_loss, N, inv_n, loss);
    SF_TRY(sf::check_launch("k_lce_loss"));
  }
  return SF_OK;
}

}  // extern "C"

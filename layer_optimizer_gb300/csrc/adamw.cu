// Fused multi-tensor AdamW for one layer (bf16 grad -> fp32 master/m/v ->
// bf16 weight), and the same moment update in the compressed d x d space of
// the sparse-projector path.
//
// The layer update is the step that SlideFormer ("An Efficient
// Heterogeneous Co-Design for Fine-Tuning on a Single GPU", technical
// summary section 2.A) runs per layer while the next layer computes, on
// flattened fp32 optimizer states with a write-back of low-precision
// weights (section 2.B).  The pages run it on the CPU; here it is an
// HBM-streaming GPU kernel.  Per element it moves 28 bytes (2 B grad, 3 x
// 4 B read and written, 2 B weight) and does ~15 flops, one sqrt and one
// divide, so HBM bandwidth bounds it.
//
// Kernel shape: a persistent grid (SMs x resident blocks) walks "tiles" of
// 4096 elements (256 threads x 2 units x 8 elements).  Each unit is one
// 16-byte grad load (8 bf16), two 16-byte loads each of master, m and v,
// the same stores, and one 16-byte bf16 weight store.  All loads of a
// thread are issued before any math so that ~220 bytes per thread are in
// flight.  Tensors whose arrays are not mutually 16-byte aligned fall back
// to a scalar loop; the (< 8 element) unaligned head and the tail of an
// aligned tensor are done by scalar code in the tensor's first/last tile.
#include <cuda_bf16.h>

#include "common.h"

namespace sf {
namespace {

constexpr int kThreads = 256;
constexpr int kUnitsPerThread = 2;
constexpr int kUnitElems = 8;
constexpr int kTileUnits = kThreads * kUnitsPerThread;     // 512
constexpr int kTileElems = kTileUnits * kUnitElems;        // 4096

struct TensorDesc {
  const uint16_t* g;
  float* p;
  float* m;
  float* v;
  uint16_t* w;       // may be null
  int64_t n;         // elements
  int64_t nvec;      // 8-element units after the head (vector mode)
  int32_t tile_begin;
  int32_t head;      // scalar elements before the first aligned unit
  int32_t tail;      // scalar elements after the last unit
  int32_t vector_mode;
};

struct LaunchArgs {
  TensorDesc t[SF_MAX_TENSORS_PER_LAUNCH];
  AdamConsts c;
  int32_t nt;
  int32_t total_tiles;
};

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}

// The AdamW element update (decoupled decay, bias-corrected moments).
__device__ __forceinline__ void adam_elem(float g, float& p, float& m, float& v,
                                          const AdamConsts& c) {
  m = fmaf(c.beta1, m, c.one_minus_beta1 * g);
  v = fmaf(c.beta2, v, c.one_minus_beta2 * (g * g));
  const float denom = sqrtf(v) / c.sqrt_bc2 + c.eps;
  p = fmaf(-c.step_size, m / denom, p * c.decay);
}

__device__ __forceinline__ void scalar_elem(const TensorDesc& d, int64_t e, const AdamConsts& c) {
  float g = bf16_to_f32(d.g[e]);
  float p = d.p[e], m = d.m[e], v = d.v[e];
  adam_elem(g, p, m, v, c);
  d.p[e] = p;
  d.m[e] = m;
  d.v[e] = v;
  if (d.w) {
    __nv_bfloat16 h = __float2bfloat16_rn(p);
    d.w[e] = *reinterpret_cast<uint16_t*>(&h);
  }
}

__global__ void __launch_bounds__(kThreads)
adamw_multi_tensor_kernel(const __grid_constant__ LaunchArgs L) {
  const AdamConsts& c = L.c;
  for (int tile = blockIdx.x; tile < L.total_tiles; tile += gridDim.x) {
    int ti = 0;
    while (ti + 1 < L.nt && L.t[ti + 1].tile_begin <= tile) ++ti;
    const TensorDesc& d = L.t[ti];
    const int lt = tile - d.tile_begin;

    if (!d.vector_mode) {
      const int64_t e0 = (int64_t)lt * kTileElems + threadIdx.x;
#pragma unroll 4
      for (int k = 0; k < kTileElems / kThreads; ++k) {
        const int64_t e = e0 + (int64_t)k * kThreads;
        if (e < d.n) scalar_elem(d, e, c);
      }
      continue;
    }

    // 128-bit path: unit u covers elements head + 8u .. head + 8u + 7.
    const uint16_t* gb = d.g + d.head;
    float* pb = d.p + d.head;
    float* mb = d.m + d.head;
    float* vb = d.v + d.head;
    uint16_t* wb = d.w ? d.w + d.head : nullptr;

    uint4 g4[kUnitsPerThread];
    float4 p4[kUnitsPerThread][2], m4[kUnitsPerThread][2], v4[kUnitsPerThread][2];
    bool ok[kUnitsPerThread];
#pragma unroll
    for (int k = 0; k < kUnitsPerThread; ++k) {
      const int64_t u = (int64_t)lt * kTileUnits + threadIdx.x + k * kThreads;
      ok[k] = u < d.nvec;
      if (ok[k]) {
        g4[k] = __ldcs(reinterpret_cast<const uint4*>(gb) + u);
        p4[k][0] = __ldcs(reinterpret_cast<const float4*>(pb) + 2 * u);
        p4[k][1] = __ldcs(reinterpret_cast<const float4*>(pb) + 2 * u + 1);
        m4[k][0] = __ldcs(reinterpret_cast<const float4*>(mb) + 2 * u);
        m4[k][1] = __ldcs(reinterpret_cast<const float4*>(mb) + 2 * u + 1);
        v4[k][0] = __ldcs(reinterpret_cast<const float4*>(vb) + 2 * u);
        v4[k][1] = __ldcs(reinterpret_cast<const float4*>(vb) + 2 * u + 1);
      }
    }
#pragma unroll
    for (int k = 0; k < kUnitsPerThread; ++k) {
      if (!ok[k]) continue;
      const int64_t u = (int64_t)lt * kTileUnits + threadIdx.x + k * kThreads;
      const uint32_t gw[4] = {g4[k].x, g4[k].y, g4[k].z, g4[k].w};
      float* pf = reinterpret_cast<float*>(&p4[k][0]);
      float* mf = reinterpret_cast<float*>(&m4[k][0]);
      float* vf = reinterpret_cast<float*>(&v4[k][0]);
      uint32_t wout[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float g0 = bf16_to_f32(gw[j] & 0xFFFFu);
        const float g1 = bf16_to_f32(gw[j] >> 16);
        adam_elem(g0, pf[2 * j], mf[2 * j], vf[2 * j], c);
        adam_elem(g1, pf[2 * j + 1], mf[2 * j + 1], vf[2 * j + 1], c);
        wout[j] = pack_bf16x2(pf[2 * j], pf[2 * j + 1]);
      }
      __stcs(reinterpret_cast<float4*>(pb) + 2 * u, p4[k][0]);
      __stcs(reinterpret_cast<float4*>(pb) + 2 * u + 1, p4[k][1]);
      __stcs(reinterpret_cast<float4*>(mb) + 2 * u, m4[k][0]);
      __stcs(reinterpret_cast<float4*>(mb) + 2 * u + 1, m4[k][1]);
      __stcs(reinterpret_cast<float4*>(vb) + 2 * u, v4[k][0]);
      __stcs(reinterpret_cast<float4*>(vb) + 2 * u + 1, v4[k][1]);
      if (wb) __stcs(reinterpret_cast<uint4*>(wb) + u, make_uint4(wout[0], wout[1], wout[2], wout[3]));
    }

    // Scalar head (first tile) and tail (last tile) of an aligned tensor.
    const int last = d.nvec > 0 ? (int)((d.nvec - 1) / kTileUnits) : 0;
    if (lt == 0 && (int)threadIdx.x < d.head) scalar_elem(d, threadIdx.x, c);
    if (lt == last && (int)threadIdx.x < d.tail)
      scalar_elem(d, d.head + d.nvec * kUnitElems + threadIdx.x, c);
  }
}

// Compressed-space AdamW: no decay, output is the step dS itself.
__global__ void __launch_bounds__(kThreads)
adamw_compressed_kernel(const float* __restrict__ S, float* __restrict__ m, float* __restrict__ v,
                        float* __restrict__ dS, int64_t n, AdamConsts c) {
  for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * kThreads) {
    const float g = S[e];
    float mm = m[e], vv = v[e];
    mm = fmaf(c.beta1, mm, c.one_minus_beta1 * g);
    vv = fmaf(c.beta2, vv, c.one_minus_beta2 * (g * g));
    const float denom = sqrtf(vv) / c.sqrt_bc2 + c.eps;
    m[e] = mm;
    v[e] = vv;
    dS[e] = c.step_size * (mm / denom);
  }
}

int blocks_per_sm() {
  static thread_local int cached = 0;
  if (!cached) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, adamw_multi_tensor_kernel, kThreads, 0) !=
            cudaSuccess || b < 1)
      b = 1;
    cached = b;
  }
  return cached;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

sf_status fill_desc(const sf_tensor& t, int index, TensorDesc* d, int32_t tile_begin) {
  if (!t.grad || !t.master || !t.exp_avg || !t.exp_avg_sq)
    return fail(SF_ERR_INVALID, "tensor %d: grad/master/exp_avg/exp_avg_sq must be non-NULL", index);
  if (!aligned(t.grad, 2) || !aligned(t.master, 4) || !aligned(t.exp_avg, 4) ||
      !aligned(t.exp_avg_sq, 4) || (t.weight && !aligned(t.weight, 2)))
    return fail(SF_ERR_INVALID, "tensor %d: element pointers must be aligned to their element size",
                index);
  d->g = static_cast<const uint16_t*>(t.grad);
  d->p = t.master;
  d->m = t.exp_avg;
  d->v = t.exp_avg_sq;
  d->w = static_cast<uint16_t*>(t.weight);
  d->n = t.numel;
  const uintptr_t ga = reinterpret_cast<uintptr_t>(t.grad);
  int64_t head = (int64_t)(((16 - (ga % 16)) % 16) / 2);
  if (head > t.numel) head = t.numel;
  const bool vec = aligned(t.master + head, 16) && aligned(t.exp_avg + head, 16) &&
                   aligned(t.exp_avg_sq + head, 16) &&
                   (!t.weight || aligned(static_cast<const uint16_t*>(t.weight) + head, 16));
  d->vector_mode = vec ? 1 : 0;
  d->tile_begin = tile_begin;
  if (vec) {
    d->head = (int32_t)head;
    d->nvec = (t.numel - head) / kUnitElems;
    d->tail = (int32_t)(t.numel - head - d->nvec * kUnitElems);
  } else {
    d->head = 0;
    d->nvec = 0;
    d->tail = 0;
  }
  return SF_OK;
}

int64_t tiles_of(const TensorDesc& d) {
  if (d.vector_mode) return d.nvec > 0 ? ceil_div<int64_t>(d.nvec, kTileUnits) : 1;
  return ceil_div<int64_t>(d.n, kTileElems);
}

}  // namespace

sf_status adamw_layer_step_impl(const sf_tensor* tensors, int n_tensors, const sf_adamw_hparams* hp,
                                int64_t step, cudaStream_t stream) {
  if (n_tensors < 0) return fail(SF_ERR_INVALID, "n_tensors < 0");
  if (n_tensors > 0 && !tensors) return fail(SF_ERR_INVALID, "tensors is NULL");
  AdamConsts c;
  SF_TRY(make_adam_consts(hp, step, true, &c));
  for (int i = 0; i < n_tensors; ++i)
    if (tensors[i].numel < 0) return fail(SF_ERR_INVALID, "tensor %d: numel < 0", i);

  static_assert(sizeof(LaunchArgs) <= 4096, "kernel parameter block too large");
  LaunchArgs L;
  const int grid_cap = sm_count() * blocks_per_sm();
  int i = 0;
  while (i < n_tensors) {
    L.c = c;
    L.nt = 0;
    int64_t tiles = 0;
    for (; i < n_tensors && L.nt < SF_MAX_TENSORS_PER_LAUNCH; ++i) {
      if (tensors[i].numel == 0) continue;
      TensorDesc d;
      SF_TRY(fill_desc(tensors[i], i, &d, (int32_t)tiles));
      const int64_t nt = tiles_of(d);
      if (tiles + nt > INT32_MAX) break;
      L.t[L.nt++] = d;
      tiles += nt;
    }
    if (L.nt == 0) continue;
    L.total_tiles = (int32_t)tiles;
    const int grid = (int)std::min<int64_t>(tiles, grid_cap);
    adamw_multi_tensor_kernel<<<grid, kThreads, 0, stream>>>(L);
    SF_TRY(check_launch("adamw_multi_tensor_kernel"));
  }
  return SF_OK;
}

sf_status adamw_compressed_impl(const float* S, float* m, float* v, float* dS, int64_t n,
                                const sf_adamw_hparams* hp, int64_t step, cudaStream_t stream) {
  if (n < 0) return fail(SF_ERR_INVALID, "d2 < 0");
  if (n > 0 && (!S || !m || !v || !dS)) return fail(SF_ERR_INVALID, "NULL array");
  AdamConsts c;
  SF_TRY(make_adam_consts(hp, step, false, &c));
  if (n == 0) return SF_OK;
  const int64_t blocks = std::min<int64_t>(ceil_div<int64_t>(n, kThreads), (int64_t)sm_count() * 8);
  adamw_compressed_kernel<<<(int)blocks, kThreads, 0, stream>>>(S, m, v, dS, n, c);
  return check_launch("adamw_compressed_kernel");
}

}  // namespace sf

extern "C" {

sf_status sf_adamw_layer_step(const sf_tensor* tensors, int n_tensors, const sf_adamw_hparams* hp,
                              int64_t step, void* stream) {
  sf::clear_error();
  return sf::adamw_layer_step_impl(tensors, n_tensors, hp, step, sf::as_stream(stream));
}

sf_status lsp_adamw_compressed(const float* S, float* m, float* v, float* dS, int64_t d2,
                               const sf_adamw_hparams* hp, int64_t step, void* stream) {
  sf::clear_error();
  return sf::adamw_compressed_impl(S, m, v, dS, d2, hp, step, sf::as_stream(stream));
}

}  // extern "C"

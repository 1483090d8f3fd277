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
// Two kernels share the element update (adam_elem):
//  - adamw_bulk_kernel, for launches with at least 2^20 16-byte aligned
//    elements: one CTA per SM, a producer warp streams grad / master / m / v
//    in 4096-element chunks into a 3-stage shared-memory ring with 1D bulk
//    copies (cp.async.bulk, mbarrier completion), 16 consumer warps update
//    from shared memory and store straight to global memory.  It keeps
//    ~168 KB per SM in flight without register staging.
//  - adamw_multi_tensor_kernel, for small launches, for the (< 8 element)
//    unaligned head and tail of each tensor, and for tensors whose arrays
//    are not mutually 16-byte aligned: a persistent grid walks 4096-element
//    tiles with 128-bit loads issued before the math (~220 bytes in flight
//    per thread), or a scalar loop.
#include <cuda_bf16.h>

#include "common.h"
#include "ptx.cuh"

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
  int32_t skip_vector;   // vector-mode tensors: only the scalar head and tail (the bulk kernel does the rest)
};

// Bulk-copy kernel: the 16-byte aligned middle of each tensor, in chunks.
constexpr int kBulkChunk = 4096;                    // elements per stage (512 threads x 8)
constexpr int kBulkStages = 3;                      // ring depth: 3 x 56 KB in flight per SM
constexpr int kBulkConsumerWarps = 16;
constexpr int kBulkStageBytes = kBulkChunk * 14;    // grad 4 KB, master / m / v 8 KB each
constexpr int kBulkOffP = kBulkChunk * 2, kBulkOffM = kBulkChunk * 6, kBulkOffV = kBulkChunk * 10;
constexpr int64_t kBulkMinElems = int64_t(1) << 20; // smaller launches keep the register-staged kernel

struct BulkTensor {
  const uint16_t* g;    // all pointers already advanced past the scalar head
  float* p;
  float* m;
  float* v;
  uint16_t* w;          // may be null
  int64_t len;          // elements of the aligned middle (a multiple of 8)
  int32_t chunk_begin;
  int32_t pad;
};

struct BulkArgs {
  BulkTensor t[SF_MAX_TENSORS_PER_LAUNCH];
  AdamConsts c;
  int32_t nt;
  int32_t total_chunks;
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
  const float denom = fmaf(sqrtf(v), c.inv_sqrt_bc2, c.eps);   // one explicit rounding
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

    if (L.skip_vector) {
      if ((int)threadIdx.x < d.head) scalar_elem(d, threadIdx.x, c);
      if ((int)threadIdx.x < d.tail) scalar_elem(d, d.head + d.nvec * kUnitElems + threadIdx.x, c);
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

// The aligned middle of every tensor, streamed through a ring of shared-memory
// stages by 1D bulk copies (cp.async.bulk): one producer warp keeps up to
// kBulkStages chunks (168 KB) of grad / master / m / v in flight per SM
// without holding them in registers; 16 consumer warps read a chunk from
// shared memory, update it and store master / m / v / weight straight to
// global memory with streaming stores.
__global__ void __launch_bounds__(32 * (kBulkConsumerWarps + 1), 1)
    adamw_bulk_kernel(const __grid_constant__ BulkArgs B) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBulkStages * kBulkStageBytes);
  uint64_t* empty = full + kBulkStages;
  int32_t* flags = reinterpret_cast<int32_t*>(empty + kBulkStages);   // [0] issued, [1] failed
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBulkStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kBulkConsumerWarps);
    }
    flags[0] = flags[1] = 0;
    fence_mbar_init_cluster();
  }
  __syncthreads();
  griddep_launch_dependents();
  griddep_wait();                // every thread: loads and stores below touch caller memory
  const int G = gridDim.x;
  const int n_my = (int)blockIdx.x < B.total_chunks ? (B.total_chunks - (int)blockIdx.x + G - 1) / G : 0;

  if (warp == kBulkConsumerWarps) {
    if (lane == 0) {
      int q = 0;
      for (; q < n_my; ++q) {
        const int s = q % kBulkStages;
        if (q >= kBulkStages && !mbar_wait(&empty[s], ((uint32_t)(q / kBulkStages) & 1u) ^ 1u)) {
          flags[1] = 1;
          break;
        }
        const int c = (int)blockIdx.x + q * G;
        int ti = 0;
        while (ti + 1 < B.nt && B.t[ti + 1].chunk_begin <= c) ++ti;
        const BulkTensor& T = B.t[ti];
        const int64_t e0 = (int64_t)(c - T.chunk_begin) * kBulkChunk;
        const uint32_t len = (uint32_t)(T.len - e0 < kBulkChunk ? T.len - e0 : kBulkChunk);
        unsigned char* st = smem + s * kBulkStageBytes;
        mbar_arrive_expect_tx(&full[s], len * 14u);
        bulk_load(st, T.g + e0, len * 2u, &full[s]);
        bulk_load(st + kBulkOffP, T.p + e0, len * 4u, &full[s]);
        bulk_load(st + kBulkOffM, T.m + e0, len * 4u, &full[s]);
        bulk_load(st + kBulkOffV, T.v + e0, len * 4u, &full[s]);
      }
      flags[0] = q;
    }
  } else {
    const AdamConsts& c = B.c;
    const uint32_t base = smem_u32(smem);
    bool failed = false;
    for (int q = 0; q < n_my; ++q) {
      const int s = q % kBulkStages;
      if (!failed && !mbar_wait(&full[s], (uint32_t)(q / kBulkStages) & 1u)) {
        failed = true;
        flags[1] = 1;
      }
      if (failed) continue;
      const int ch = (int)blockIdx.x + q * G;
      int ti = 0;
      while (ti + 1 < B.nt && B.t[ti + 1].chunk_begin <= ch) ++ti;
      const BulkTensor& T = B.t[ti];
      const int64_t e0 = (int64_t)(ch - T.chunk_begin) * kBulkChunk;
      const int64_t len = T.len - e0 < kBulkChunk ? T.len - e0 : kBulkChunk;
      const int t = threadIdx.x;
      if (8 * t < len) {
        const uint32_t st = base + (uint32_t)(s * kBulkStageBytes);
        uint4 g4;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(g4.x), "=r"(g4.y), "=r"(g4.z), "=r"(g4.w)
                     : "r"(st + 16u * t));
        float4 p4[2] = {lds_f4(st + kBulkOffP + 32u * t), lds_f4(st + kBulkOffP + 32u * t + 16u)};
        float4 m4[2] = {lds_f4(st + kBulkOffM + 32u * t), lds_f4(st + kBulkOffM + 32u * t + 16u)};
        float4 v4[2] = {lds_f4(st + kBulkOffV + 32u * t), lds_f4(st + kBulkOffV + 32u * t + 16u)};
        const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
        float* pf = reinterpret_cast<float*>(&p4[0]);
        float* mf = reinterpret_cast<float*>(&m4[0]);
        float* vf = reinterpret_cast<float*>(&v4[0]);
        uint32_t wout[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          adam_elem(bf16_to_f32(gw[j] & 0xFFFFu), pf[2 * j], mf[2 * j], vf[2 * j], c);
          adam_elem(bf16_to_f32(gw[j] >> 16), pf[2 * j + 1], mf[2 * j + 1], vf[2 * j + 1], c);
          wout[j] = pack_bf16x2(pf[2 * j], pf[2 * j + 1]);
        }
        const int64_t o = e0 + 8 * t;
        __stcs(reinterpret_cast<float4*>(T.p + o), p4[0]);
        __stcs(reinterpret_cast<float4*>(T.p + o) + 1, p4[1]);
        __stcs(reinterpret_cast<float4*>(T.m + o), m4[0]);
        __stcs(reinterpret_cast<float4*>(T.m + o) + 1, m4[1]);
        __stcs(reinterpret_cast<float4*>(T.v + o), v4[0]);
        __stcs(reinterpret_cast<float4*>(T.v + o) + 1, v4[1]);
        if (T.w) __stcs(reinterpret_cast<uint4*>(T.w + o), make_uint4(wout[0], wout[1], wout[2], wout[3]));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_local(&empty[s]);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && flags[1]) {
    // a wait ran out: let the copies still in flight land (bounded) before exit
    const int issued = flags[0];
    for (int q = issued > kBulkStages ? issued - kBulkStages : 0; q < issued; ++q)
      mbar_wait(&full[q % kBulkStages], (uint32_t)(q / kBulkStages) & 1u);
  }
}

// Compressed-space AdamW: no decay, output is the step dS itself.
__global__ void __launch_bounds__(kThreads)
adamw_compressed_kernel(const float* __restrict__ S, float* __restrict__ m, float* __restrict__ v,
                        float* __restrict__ dS, int64_t n, AdamConsts c) {
  griddep_launch_dependents();
  griddep_wait();                // S comes from the compress kernels
  for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * kThreads) {
    const float g = S[e];
    float mm = m[e], vv = v[e];
    mm = fmaf(c.beta1, mm, c.one_minus_beta1 * g);
    vv = fmaf(c.beta2, vv, c.one_minus_beta2 * (g * g));
    const float denom = fmaf(sqrtf(vv), c.inv_sqrt_bc2, c.eps);
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
  // Arrays in pinned host memory (or anywhere but this device's memory) are
  // updated in place with the register-staged kernel's plain loads and
  // stores (zero-copy over the host link); the bulk kernel's shared-memory
  // copies read only this device's own memory.
  bool host_resident = false;
  for (int i = 0; i < n_tensors && !host_resident; ++i) {
    const sf_tensor& t = tensors[i];
    if (t.numel == 0) continue;
    if (!on_current_device(t.master) || !on_current_device(t.grad) || !on_current_device(t.exp_avg) ||
        !on_current_device(t.exp_avg_sq))
      host_resident = true;
  }
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
    // Large launches: the aligned middles go through the bulk-copy kernel and
    // the register-staged kernel only does scalar heads / tails and tensors
    // that are not mutually 16-byte aligned.
    int64_t vec_elems = 0;
    for (int t = 0; t < L.nt; ++t)
      if (L.t[t].vector_mode) vec_elems += L.t[t].nvec * kUnitElems;
    L.skip_vector = !host_resident && vec_elems >= kBulkMinElems ? 1 : 0;
    if (L.skip_vector) {
      BulkArgs B;
      B.c = c;
      B.nt = 0;
      int64_t chunks = 0;
      bool scalar_work = false;
      int64_t rtiles = 0;
      for (int t = 0; t < L.nt; ++t) {
        TensorDesc& d = L.t[t];
        d.tile_begin = (int32_t)rtiles;
        if (!d.vector_mode) {
          rtiles += tiles_of(d);
          scalar_work = true;
          continue;
        }
        rtiles += 1;
        if (d.head || d.tail) scalar_work = true;
        if (d.nvec == 0) continue;
        BulkTensor& T = B.t[B.nt++];
        T.g = d.g + d.head;
        T.p = d.p + d.head;
        T.m = d.m + d.head;
        T.v = d.v + d.head;
        T.w = d.w ? d.w + d.head : nullptr;
        T.len = d.nvec * kUnitElems;
        T.chunk_begin = (int32_t)chunks;
        T.pad = 0;
        chunks += ceil_div<int64_t>(T.len, kBulkChunk);
      }
      B.total_chunks = (int32_t)chunks;
      static_assert(sizeof(BulkArgs) <= 4096, "kernel parameter block too large");
      const size_t smem = (size_t)kBulkStages * kBulkStageBytes + 2 * kBulkStages * 8 + 8;
      SF_TRY(allow_dynamic_smem(reinterpret_cast<const void*>(&adamw_bulk_kernel), smem));
      if (B.nt > 0) {
        const int grid = (int)std::min<int64_t>(chunks, sm_count());
        SF_CUDA_TRY(launch_pdl(adamw_bulk_kernel, dim3(grid), dim3(32 * (kBulkConsumerWarps + 1)), smem, stream, B),
                    "launch adamw_bulk_kernel");
      }
      if (!scalar_work) continue;
      L.total_tiles = (int32_t)rtiles;
      adamw_multi_tensor_kernel<<<(int)std::min<int64_t>(rtiles, grid_cap), kThreads, 0, stream>>>(L);
      SF_TRY(check_launch("adamw_multi_tensor_kernel"));
      continue;
    }
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
  SF_CUDA_TRY(launch_pdl(adamw_compressed_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, S, m, v, dS, n, c),
              "launch adamw_compressed_kernel");
  return SF_OK;
}

// A wait on an mbarrier that nothing arrives on, bounded by `limit` cycles:
// runs out, records kDevErrTimeout and returns (the path every bounded wait
// in the library takes when its copies never land).
__global__ void k_test_wait_runs_out(long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init_cluster();
  mbar_wait_limit(&bar, 0, limit);
}

int read_and_clear_device_error_adamw() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof z);
  return v;
}

}  // namespace sf

extern "C" {

sf_status sf_adamw_layer_step(const sf_tensor* tensors, int n_tensors, const sf_adamw_hparams* hp,
                              int64_t step, void* stream) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("sf_adamw_layer_step");
  return sf::adamw_layer_step_impl(tensors, n_tensors, hp, step, sf::as_stream(stream));
}

sf_status lsp_adamw_compressed(const float* S, float* m, float* v, float* dS, int64_t d2,
                               const sf_adamw_hparams* hp, int64_t step, void* stream) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("lsp_adamw_compressed");
  return sf::adamw_compressed_impl(S, m, v, dS, d2, hp, step, sf::as_stream(stream));
}

sf_status sf_test_device_wait_runs_out(int64_t limit_cycles, void* stream) {
  sf::clear_error();
  if (limit_cycles < 1 || limit_cycles > 4000000000LL)
    return sf::fail(SF_ERR_INVALID, "limit_cycles must be in [1, 4e9]");
  sf::k_test_wait_runs_out<<<1, 32, 0, sf::as_stream(stream)>>>((long long)limit_cycles);
  return sf::check_launch("k_test_wait_runs_out");
}

}  // extern "C"

// Tensor-memory gather rate: the other on-chip source the projector kernels
// could gather from.
//
// The compress and decompress kernels (lsp.cu) read their dense operand at
// rows chosen by projector indices; in shared memory every such multiply-add
// costs a 4-byte lane load out of the SM's 128-byte-per-clock crossbar
// (sf_bench_gather_rate measures that roof).  On sm_103a each SM also has
// 256 KB of tensor memory (TMEM: 128 lanes x 512 32-bit columns) that warps
// read with tcgen05.ld, a warp reaching the 32 lanes of its quarter (warp id
// mod 4) at a column address it chooses at run time.  Holding the dense
// operand there with lanes along its contiguous dimension turns a gathered
// row into one column load, so this kernel measures how fast such loads run
// when their columns are chosen per step, the way a gather would use them:
//   x        columns per load (tcgen05.ld.32x32b.x1, .x2 or .x4)
//   entries  1: each load's column and value come from a shared-memory entry
//            list (an 8-byte broadcast per load, as a gather kernel reads its
//            projector entries); 0: computed in registers (TMEM alone)
// Each step issues 8 loads, waits for them (tcgen05.wait::ld) and does
// 8 * x multiply-adds per thread.  One CTA of 16 warps per SM owns all 512
// columns (allocated and released inside the launch).  No global memory
// traffic in the loop.  A third probe times row gathers straight from L2.
#include "common.h"
#include "ptx.cuh"

namespace sf {
namespace {

constexpr int kTmThreads = 512;
constexpr int kTmCols = 512;
constexpr int kTmEntries = 2048;
constexpr int kTmBatch = 8;
// shared memory requested per CTA: the entry list plus padding, so that two
// CTAs never share an SM (each allocates every TMEM column)
constexpr size_t kTmSmem = 128 * 1024;

__device__ __forceinline__ void tm_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tm_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tm_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tm_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tm_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tm_st4(uint32_t taddr, float a, float b, float c, float d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}
__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// X consecutive 32-bit columns of this thread's lane at `taddr`.
template <int X>
__device__ __forceinline__ void tm_ld(uint32_t taddr, float (&r)[X]) {
  if constexpr (X == 1) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=f"(r[0]) : "r"(taddr));
  } else if constexpr (X == 2) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];" : "=f"(r[0]), "=f"(r[1]) : "r"(taddr));
  } else {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3])
                 : "r"(taddr));
  }
}

// Waits for this thread's outstanding tcgen05.ld; the registers pass through
// the statement so no use of them can be scheduled before the wait.
template <int X>
__device__ __forceinline__ void tm_wait_ld(float (&r)[kTmBatch][X]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int u = 0; u < kTmBatch; ++u)
#pragma unroll
    for (int j = 0; j < X; ++j) asm volatile("" : "+f"(r[u][j]));
}

template <int X, bool kEntries>
__global__ void __launch_bounds__(kTmThreads, 1) k_tmem_rate(int64_t iters, float* __restrict__ sink) {
  extern __shared__ __align__(16) unsigned char smem[];
  int2* ent = reinterpret_cast<int2*>(smem);
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3;
  if (warp == 0) {
    tm_alloc(smem_u32(&tmem_slot), kTmCols);
    tm_relinquish();
  }
  // columns stepped in units of X so every load stays inside the 512 columns
  constexpr int kSlots = kTmCols / X;
  for (int e = threadIdx.x; e < kTmEntries; e += blockDim.x) {
    const uint32_t h = (uint32_t)e * 2654435761u + blockIdx.x;
    ent[e] = make_int2((int)(((h >> 9) % kSlots) * X), __float_as_int(1.0f / (float)(1 + (e & 7))));
  }
  tm_fence_before();
  __syncthreads();
  tm_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
  if (warp < 4) {
    for (int c = 0; c < kTmCols; c += 4) {
      const float b = (float)((lane * 7 + c) & 1023) * (1.0f / 1024.0f);
      tm_st4(lane_base + (uint32_t)c, b, b + 0.25f, b + 0.5f, b + 0.75f);
    }
    tm_wait_st();
  }
  tm_fence_before();
  __syncthreads();
  tm_fence_after();

  const uint32_t ent_base = smem_u32(ent);
  float acc[X];
#pragma unroll
  for (int j = 0; j < X; ++j) acc[j] = 0.0f;
  uint32_t e = (uint32_t)warp * 128u;
  uint32_t col_r = (uint32_t)warp * 37u;
  for (int64_t it = 0; it < iters; ++it) {
    float r[kTmBatch][X];
    float v[kTmBatch];
#pragma unroll
    for (int u = 0; u < kTmBatch; ++u) {
      uint32_t col;
      if constexpr (kEntries) {
        const int2 en = lds_i2(ent_base + 8u * ((e + (uint32_t)u) & (kTmEntries - 1)));
        col = (uint32_t)en.x;
        v[u] = __int_as_float(en.y);
      } else {
        col = ((col_r + 97u * (uint32_t)u) % (uint32_t)kSlots) * X;
        v[u] = 1.0f / (float)(1 + u);
      }
      tm_ld<X>(lane_base + col, r[u]);
    }
    tm_wait_ld<X>(r);
#pragma unroll
    for (int u = 0; u < kTmBatch; ++u)
#pragma unroll
      for (int j = 0; j < X; ++j) acc[j] = fmaf(v[u], r[u][j], acc[j]);
    e += kTmBatch;
    col_r += 13u;
  }
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < X; ++j) s += acc[j];
  sink[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
  tm_fence_before();
  __syncthreads();
  if (warp == 0) {
    tm_fence_after();
    tm_dealloc(tmem, kTmCols);
  }
}

template <int X, bool kEntries>
sf_status launch_tmem_rate(int ctas, int64_t iters, float* sink, cudaStream_t s) {
  auto kern = k_tmem_rate<X, kEntries>;
  SF_TRY(allow_dynamic_smem(reinterpret_cast<const void*>(kern), kTmSmem));
  kern<<<(unsigned)ctas, kTmThreads, kTmSmem, s>>>(iters, sink);
  return check_launch("k_tmem_rate");
}

// L2 row-gather rate: the third source a gather can read from.  Each warp
// reads 512-byte rows (one 16-byte load per lane) of a caller buffer at rows
// chosen per load, 16 loads in flight per lane, and does 4 multiply-adds per
// loaded float4.  With the buffer smaller than L2 and warmed, the loop
// measures how fast the SMs can gather rows straight from L2.
constexpr int kL2Unroll = 16;
__global__ void __launch_bounds__(256, 2) k_l2_gather_rate(const float4* __restrict__ buf, uint32_t rows,
                                                           int64_t iters, float* __restrict__ sink) {
  const int lane = threadIdx.x & 31;
  const uint32_t gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  uint32_t h = gw * 2654435761u + 12345u;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t it = 0; it < iters; ++it) {
    float4 x[kL2Unroll];
#pragma unroll
    for (int u = 0; u < kL2Unroll; ++u) {
      h = h * 1664525u + 1013904223u;
      const uint32_t row = (h >> 8) % rows;
      x[u] = buf[(size_t)row * 32 + lane];
    }
#pragma unroll
    for (int u = 0; u < kL2Unroll; ++u) {
      const float q = 1.0f / (float)(1 + u);
      acc.x = fmaf(q, x[u].x, acc.x);
      acc.y = fmaf(q, x[u].y, acc.y);
      acc.z = fmaf(q, x[u].z, acc.z);
      acc.w = fmaf(q, x[u].w, acc.w);
    }
  }
  sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = acc.x + acc.y + acc.z + acc.w;
}

}  // namespace
}  // namespace sf

extern "C" {

sf_status sf_bench_l2_gather_rate(int32_t ctas, int64_t iters, const float* buf, int64_t rows, float* sink,
                                  void* stream) {
  sf::clear_error();
  if (ctas < 1 || iters < 1 || !sink || !buf || rows < 1 || rows > (int64_t)UINT32_MAX)
    return sf::fail(SF_ERR_INVALID, "ctas, iters and rows must be >= 1 (rows < 2^32), buf and sink non-NULL");
  if (reinterpret_cast<uintptr_t>(buf) % 16) return sf::fail(SF_ERR_INVALID, "buf must be 16-byte aligned");
  sf::k_l2_gather_rate<<<(unsigned)ctas, 256, 0, sf::as_stream(stream)>>>(reinterpret_cast<const float4*>(buf),
                                                                         (uint32_t)rows, iters, sink);
  return sf::check_launch("k_l2_gather_rate");
}

sf_status sf_bench_tmem_rate(int32_t ctas, int64_t iters, int32_t x, int32_t entries, float* sink, void* stream) {
  sf::clear_error();
  if (ctas < 1 || iters < 1 || !sink) return sf::fail(SF_ERR_INVALID, "ctas and iters must be >= 1, sink non-NULL");
  if (x != 1 && x != 2 && x != 4) return sf::fail(SF_ERR_INVALID, "x must be 1, 2 or 4 (got %d)", x);
  cudaStream_t s = sf::as_stream(stream);
  const bool e = entries != 0;
  if (x == 1) return e ? sf::launch_tmem_rate<1, true>(ctas, iters, sink, s) : sf::launch_tmem_rate<1, false>(ctas, iters, sink, s);
  if (x == 2) return e ? sf::launch_tmem_rate<2, true>(ctas, iters, sink, s) : sf::launch_tmem_rate<2, false>(ctas, iters, sink, s);
  return e ? sf::launch_tmem_rate<4, true>(ctas, iters, sink, s) : sf::launch_tmem_rate<4, false>(ctas, iters, sink, s);
}

}  // extern "C"

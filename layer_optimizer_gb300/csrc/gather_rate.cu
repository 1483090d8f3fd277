// Shared-memory gather rate: the second roof of the projector kernels.
//
// The compress and decompress kernels (lsp.cu) are sparse products: every
// multiply-add reads its dense operand from a shared-memory tile at a row
// chosen by a projector index, so besides HBM they are bounded by how fast
// the SMs can do such gathered multiply-adds.  This kernel measures that
// rate with the gather kernels' inner loop and nothing else: a tile of 128
// rows x 128 fp32 columns and a list of (row, value) entries in shared
// memory, each lane owning 4 columns, two entries per step (two 8-byte entry
// loads, two 16-byte tile loads at dynamic rows, 8 multiply-adds), 16 warps
// per SM as in the gather kernels.  No global memory traffic in the loop.
#include "common.h"
#include "ptx.cuh"

namespace sf {
namespace {

constexpr int kRateThreads = 512;
constexpr int kRateRows = 128, kRateRowBytes = 128 * 4, kRateEntries = 2048;

__global__ void __launch_bounds__(kRateThreads, 1) k_gather_rate(int64_t iters, float* __restrict__ sink) {
  extern __shared__ __align__(16) unsigned char smem[];
  float* tile = reinterpret_cast<float*>(smem);
  int2* ent = reinterpret_cast<int2*>(smem + kRateRows * kRateRowBytes);
  for (int i = threadIdx.x; i < kRateRows * 128; i += blockDim.x) tile[i] = (float)(i & 1023) * (1.0f / 1024.0f);
  for (int e = threadIdx.x; e < kRateEntries; e += blockDim.x) {
    const uint32_t h = (uint32_t)e * 2654435761u + blockIdx.x;     // scattered rows, fixed by e
    ent[e] = make_int2((int)((h >> 9) % kRateRows), __float_as_int(1.0f / (float)(1 + (e & 7))));
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tile_lane = smem_u32(tile) + 16u * (uint32_t)lane;
  const uint32_t ent_base = smem_u32(ent);
  float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
  uint32_t e = (uint32_t)warp * 128u;
  for (int64_t it = 0; it < iters; ++it, e += 2u) {
    const uint32_t ei = e & (kRateEntries - 2);
    const int2 en0 = lds_i2(ent_base + 8u * ei);
    const int2 en1 = lds_i2(ent_base + 8u * ei + 8u);
    const float4 x0 = lds_f4(tile_lane + (uint32_t)en0.x * (uint32_t)kRateRowBytes);
    const float4 x1 = lds_f4(tile_lane + (uint32_t)en1.x * (uint32_t)kRateRowBytes);
    const float v0 = __int_as_float(en0.y), v1 = __int_as_float(en1.y);
    a0 = fmaf(v1, x1.x, fmaf(v0, x0.x, a0));
    a1 = fmaf(v1, x1.y, fmaf(v0, x0.y, a1));
    a2 = fmaf(v1, x1.z, fmaf(v0, x0.z, a2));
    a3 = fmaf(v1, x1.w, fmaf(v0, x0.w, a3));
  }
  sink[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = a0 + a1 + a2 + a3;
}

}  // namespace
}  // namespace sf

extern "C" {

sf_status sf_bench_gather_rate(int32_t ctas, int64_t iters, float* sink, void* stream) {
  sf::clear_error();
  if (ctas < 1 || iters < 1 || !sink) return sf::fail(SF_ERR_INVALID, "ctas and iters must be >= 1, sink non-NULL");
  const size_t smem = (size_t)sf::kRateRows * sf::kRateRowBytes + (size_t)sf::kRateEntries * 8;
  SF_TRY(sf::allow_dynamic_smem(reinterpret_cast<const void*>(&sf::k_gather_rate), smem));
  sf::k_gather_rate<<<(unsigned)ctas, sf::kRateThreads, smem, sf::as_stream(stream)>>>(iters, sink);
  return sf::check_launch("k_gather_rate");
}

}  // extern "C"

// Tensor-core GEMM on the 5th-generation tensor cores: C (fp32) = alpha A B^T
// (+ C) with A [M x K] and B [N x K] in bf16, each stored either K-major
// (row-major [M][K], [N][K]) or MN-major (row-major [K][M], [K][N]: the
// transposed matrix), so products like G W or G^T H need no transposed copy.
//
// The dense products of the fused linear cross-entropy (logits, and the two
// gradient products) are real dense contractions, so they run here rather
// than on CUDA cores.  Pairs of CTAs (a cluster of two, one per SM of a
// TPC) walk the 256 x 256 tiles of C in a persistent grid, and each pair
// computes its tile with the pair form of the MMA (cta_group::2, M 256):
// every CTA holds 128 rows of A and 128 rows of B per K slab, the MMA reads
// both halves across the pair, and each CTA's TMEM receives its 128 rows of
// the 256 x 256 accumulator.  Per SM that is half the B tile in shared
// memory and half its shared-memory read traffic, compared with one CTA
// computing 128 x 256 alone, which leaves room for a 6-deep ring.  In each
// CTA:
//   warp 0       TMA producer: 64-wide K slabs of its A rows (128 x 64) and
//                B rows (128 x 64) into a 6-stage ring, 128-byte swizzled
//                (a K-major operand as one 128-row box, an MN-major one as
//                two boxes of 64 x 64); both CTAs' copies complete on the
//                first CTA's stage barrier;
//   warp 1       allocates 512 TMEM columns with its peer (two accumulators
//                of 256 fp32 columns); in the first CTA one elected thread
//                issues tcgen05.mma (M 256, N 256, K 16, bf16 in, fp32
//                accumulate), four per slab, into the accumulator both
//                epilogues have released; tcgen05.commit frees a stage in
//                both CTAs when its MMAs are done and, after a tile's last
//                slab, hands the accumulator to both epilogues;
//   warps 2..5   epilogue: each reads its 32 TMEM lanes (rows) with
//                tcgen05.ld and writes (or reduce-adds into) C by tensor
//                stores from shared memory, while the next tile's MMAs run
//                into the other accumulator.
// Every wait is bounded: a wait that runs out records an error for
// sf_sync_status, and the CTAs still release their TMEM before they exit.
// Sums over K run in slab order on the tensor cores; results are
// deterministic for a given shape.
#include <cuda_bf16.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "common.h"
#include "ptx.cuh"

namespace sf {
namespace {

constexpr int kPair = 2;                       // CTAs per tile (cta_group::2)
constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 6;
constexpr int kBRows = kBN / kPair;            // rows of B held by one CTA
constexpr int kStageA = kBM * kBK * 2;         // 16 KB
constexpr int kStageB = kBRows * kBK * 2;      // 16 KB
constexpr int kStageBytes = kStageA + kStageB;
constexpr int kMnBox = 64 * kBK * 2;           // an MN-major box: 64 MN x 64 K bf16 = 8 KB
constexpr int kTmemCols = 256;                 // one accumulator; two are allocated
constexpr int kGemmThreads = 192;
constexpr int kStagingBytes = 4 * 2 * 4096;    // epilogue: 4 warps x 2 boxes of 32 x 32 fp32
constexpr size_t kGemmSmem = (size_t)kStages * kStageBytes + kStagingBytes + 1024 + 256;

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator
// (bits 4-5 = 1), A and B bf16 (bits 7-9 and 10-12 = 1), A and B K-major
// (bits 15, 16 = 0; set per launch for an MN-major operand), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28 (M = 256: the pair's rows).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)((kPair * kBM) >> 4) << 24);

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes (64 bf16 of K), 8-row atoms of
// 1024 bytes (stride-dimension offset), descriptor version 1, layout type 2.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  uint64_t d = (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading-dimension offset (unused when swizzled)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride-dimension offset: 1024 bytes
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)2 << 61;                 // 128-byte swizzle
  return d;
}

// The same for an MN-major operand tile: TMA boxes of 64 MN-contiguous
// elements (128 bytes) by 64 K rows, 128-byte swizzled, two of them side by
// side for 128 rows of MN.  The canonical MN-major layout takes the offset
// between 64-element MN blocks as the leading-dimension offset (one box,
// 8192 bytes) and between 8-row K groups as the stride-dimension offset
// (1024 bytes); a K-16 step advances the start by 16 rows = 2048 bytes.
__device__ __forceinline__ uint64_t umma_desc_mn_sw128(uint32_t smem_addr) {
  uint64_t d = (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(kMnBox >> 4) << 16;     // leading-dimension offset: next 64 MN elements
  d |= (uint64_t)(1024 >> 4) << 32;       // stride-dimension offset: next 8 K rows
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// TMEM allocation of the CTA pair: one warp of each CTA issues these
// together (the pair form requires both).
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A B^T for one K-16 step over the pair (M 256: A rows from
// both CTAs' shared memory at the descriptor's offset, B likewise, D rows
// 0-127 into this CTA's TMEM and 128-255 into the peer's); accumulate = 0
// overwrites D.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the barrier at shared offset `mbar` in both CTAs of the pair
// once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void tc_commit_pair(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          mbar),
      "h"((uint16_t)3)
      : "memory");
}

// 2D tiled TMA load into this CTA's shared memory whose completion is
// counted on the barrier at shared::cluster address `bar` (the pair form
// lets it be the first CTA's barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                                 int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// The same with a 3D box (an MN-major operand: 64 MN x 64 K x two
// 64-element MN blocks, stored block after block).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// Arrival on a barrier of another CTA of the cluster, ordering this
// thread's earlier accesses (TMEM reads included, after
// tcgen05.fence::before_thread_sync) at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote_release(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Bounded wait with cluster-scope acquire (arrivals from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  auto test = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (test()) return true;
  const long long t0 = clock64();
  for (;;) {
    if (test()) return true;
    if (clock64() - t0 > kWaitLimitCycles) {
      atomicOr(&g_device_error, kDevErrTimeout);
      return false;
    }
  }
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Tensor store / reduce-add of a shared-memory box into global memory
// (bulk async group of this thread), and the group waits.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   map),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void sts_f4(uint32_t a, float x, float y, float z, float w) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x), "f"(y), "f"(z), "f"(w) : "memory");
}

struct TcGemmArgs {
  float* C;
  int64_t ldc;
  int32_t M, N, K;
  float alpha;
  int32_t accumulate;    // 1: C += alpha A B^T, 0: C = alpha A B^T
  int32_t vec;           // C rows 16-byte aligned (float4 epilogue)
  int32_t tma;           // C written by tensor stores (reduce-add when accumulating) from shared memory
  int32_t n_fast;        // tile order: n fastest (A is the larger operand) or m fastest
  int32_t a_mn, b_mn;    // operand stored MN-major ([K][M], [K][N]) instead of K-major:
                         // 1 loaded as two 2D boxes, 2 as one 3D box (MN a multiple of 64)
  float2* row_stats;     // optional [M][n_tiles]: per row and column tile, (max, sum exp(c - max)) of C
};

// Folds 32 values of a row into a running (max, sum of exp(x - max)):
// the chunk's maximum first, then one rescale of the running sum.
__device__ __forceinline__ void fold_row_stats(const float (&x)[32], int valid, float& m, float& s) {
  float cm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j < valid) cm = fmaxf(cm, x[j]);
  if (cm == -INFINITY) return;
  const float mn = fmaxf(m, cm);
  float acc = m == -INFINITY ? 0.0f : s * expf(m - mn);
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j < valid) acc += expf(x[j] - mn);
  m = mn;
  s = acc;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
              const __grid_constant__ CUtensorMap map_c, const TcGemmArgs g) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // [ring: kStages x (A 16 KB + B 16 KB)] [epilogue staging: 4 warps x 2 x 4 KB] [barriers]
  unsigned char* staging = smem + (size_t)kStages * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + kStagingBytes);   // used in the first CTA
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;     // [2] accumulator buffer b holds a finished tile
  uint64_t* tempty = tfull + 2;          // [2] both CTAs have read buffer b out (first CTA)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t empty_a = smem_u32(empty), tfull_a = smem_u32(tfull);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();              // 0: issues the MMAs, 1: its peer
  const int pair = blockIdx.x / kPair, n_pairs = gridDim.x / kPair;
  const int nk = (g.K + kBK - 1) / kBK;
  const int m_tiles = (g.M + kPair * kBM - 1) / (kPair * kBM);   // 256-row tiles
  const int n_tiles = (g.N + kBN - 1) / kBN;
  const int tiles = m_tiles * n_tiles;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);            // the first CTA's producer arrives, both CTAs' copies complete it
      mbar_init(&empty[s], 1);           // the MMA commit arrives in both CTAs
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4 * kPair);  // one arrival per epilogue warp of the pair
    }
    fence_mbar_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();                        // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // tiles t = pair, + n_pairs, ...; the index runs fastest along the
  // dimension whose operand is the smaller one, so the pairs working at the
  // same time share the tile of the larger operand and it streams from
  // memory about once, while the smaller one is re-read from L2
  if (warp == 0) {
    if (lane == 0) {
      griddep_wait();
      const uint32_t full_lead = cluster_addr(smem_u32(full), 0);
      int s = 0, issued = 0;
      uint32_t pass = 0;
      bool failed = false;
      for (int t = pair; t < tiles && !failed; t += n_pairs) {
        const int mt = g.n_fast ? t / n_tiles : t % m_tiles, nt = g.n_fast ? t % n_tiles : t / m_tiles;
        const int m0 = mt * (kPair * kBM) + (int)rank * kBM;
        const int nb = nt * kBN + (int)rank * kBRows;
        for (int kb = 0; kb < nk; ++kb) {
          if (issued >= kStages && !mbar_wait_cluster(&empty[s], pass ^ 1u)) {
            failed = true;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(kPair * kStageBytes));
          const uint32_t st = smem_base + (uint32_t)s * kStageBytes;
          const uint32_t bar = full_lead + 8u * (uint32_t)s;
          if (g.a_mn == 2) {
            tma_load_3d_pair(st, &map_a, bar, 0, kb * kBK, m0 >> 6);
          } else if (g.a_mn) {
            tma_load_2d_pair(st, &map_a, bar, m0, kb * kBK);
            tma_load_2d_pair(st + kMnBox, &map_a, bar, m0 + 64, kb * kBK);
          } else {
            tma_load_2d_pair(st, &map_a, bar, kb * kBK, m0);
          }
          if (g.b_mn == 2) {
            tma_load_3d_pair(st + kStageA, &map_b, bar, 0, kb * kBK, nb >> 6);
          } else if (g.b_mn) {
            tma_load_2d_pair(st + kStageA, &map_b, bar, nb, kb * kBK);
            tma_load_2d_pair(st + kStageA + kMnBox, &map_b, bar, nb + 64, kb * kBK);
          } else {
            tma_load_2d_pair(st + kStageA, &map_b, bar, kb * kBK, nb);
          }
          ++issued;
          if (++s == kStages) {
            s = 0;
            pass ^= 1u;
          }
        }
      }
      // the copies of the last stages (both CTAs') have landed before the
      // pair can exit: immediate when the MMA thread consumed them, bounded
      // otherwise
      if (rank == 0)
        for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
          mbar_wait_cluster(&full[j % kStages], (uint32_t)(j / kStages) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // K-16 step in descriptor units (16 bytes): 32 bytes along a K-major
      // row, 16 rows of 128 bytes down an MN-major box
      const uint32_t a_step = g.a_mn ? 128u : 2u, b_step = g.b_mn ? 128u : 2u;
      const uint32_t idesc = kIdesc | ((g.a_mn ? 1u : 0u) << 15) | ((g.b_mn ? 1u : 0u) << 16);
      int s = 0, j = 0;
      uint32_t pass = 0;
      bool failed = false;
      for (int t = pair; t < tiles && !failed; t += n_pairs, ++j) {
        const int b = j & 1;
        const uint32_t use = (uint32_t)(j >> 1);
        // both epilogues have read this accumulator buffer out (its previous use)
        if (use > 0 && !mbar_wait_cluster(&tempty[b], (use - 1u) & 1u)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(b * kTmemCols);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_cluster(&full[s], pass)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_base + (uint32_t)s * kStageBytes;
          const uint64_t adesc = g.a_mn ? umma_desc_mn_sw128(a_addr) : umma_desc_sw128(a_addr);
          const uint64_t bdesc = g.b_mn ? umma_desc_mn_sw128(a_addr + kStageA) : umma_desc_sw128(a_addr + kStageA);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc_mma(d_tmem, adesc + a_step * (uint32_t)k, bdesc + b_step * (uint32_t)k, idesc, (kb | k) != 0 ? 1u : 0u);
          tc_commit_pair(empty_a + 8u * (uint32_t)s);
          if (++s == kStages) {
            s = 0;
            pass ^= 1u;
          }
        }
        tc_commit_pair(tfull_a + 8u * (uint32_t)b);
      }
    }
  } else {
    // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 = rows of this
    // CTA's half of the tile
    const int quarter = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const uint32_t stg = smem_u32(staging) + (uint32_t)(warp - 2) * 8192u;
    const uint32_t tempty_lead = cluster_addr(smem_u32(tempty), 0);
    int j = 0, boxes = 0;
    for (int t = pair; t < tiles; t += n_pairs, ++j) {
      const int mt = g.n_fast ? t / n_tiles : t % m_tiles, nt = g.n_fast ? t % n_tiles : t / m_tiles;
      const int m0 = mt * (kPair * kBM) + (int)rank * kBM, n0 = nt * kBN;
      const int b = j & 1;
      if (!mbar_wait_cluster(&tfull[b], (uint32_t)(j >> 1) & 1u)) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(b * kTmemCols) + lane_off;
      const int row = m0 + 32 * quarter + lane;
      if (g.tma) {
        // 32 x 32 boxes through two 4 KB staging buffers per warp, 128-byte
        // swizzled to match the store's tensor map (conflict-free 16-byte
        // writes); one thread stores or reduce-adds each box, and a buffer
        // is rewritten only once its previous store has read it
        const int row0 = m0 + 32 * quarter;
        float rm = -INFINITY, rs = 0.0f;
#pragma unroll 1
        for (int ci = 0; ci < kBN / 32; ++ci, ++boxes) {
          uint32_t r[32];
          tmem_ld32(acc + (uint32_t)(32 * ci), r);
          tmem_ld_wait();
          if (g.row_stats) {
            float x[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) x[jj] = g.alpha * __uint_as_float(r[jj]);
            fold_row_stats(x, min(32, g.N - (n0 + 32 * ci)), rm, rs);
          }
          const uint32_t buf = stg + (uint32_t)(boxes & 1) * 4096u;
          if (boxes >= 2) {
            if (lane == 0) bulk_wait_read_1();
            __syncwarp();
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            sts_f4(buf + (uint32_t)lane * 128u + (uint32_t)((q ^ (lane & 7)) * 16), g.alpha * __uint_as_float(r[4 * q]),
                   g.alpha * __uint_as_float(r[4 * q + 1]), g.alpha * __uint_as_float(r[4 * q + 2]),
                   g.alpha * __uint_as_float(r[4 * q + 3]));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (row0 < g.M && n0 + 32 * ci < g.N) {
              if (g.accumulate) tma_reduce_add_2d(&map_c, buf, n0 + 32 * ci, row0);
              else tma_store_2d(&map_c, buf, n0 + 32 * ci, row0);
            }
            bulk_commit();
          }
          __syncwarp();
        }
        if (g.row_stats && row < g.M) g.row_stats[(int64_t)row * n_tiles + nt] = make_float2(rm, rs);
      } else {
        const bool row_on = row < g.M;
        float* crow = g.C + (int64_t)row * g.ldc;
        float rm = -INFINITY, rs = 0.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(acc + (uint32_t)c0, r);
          tmem_ld_wait();
          const int col0 = n0 + c0;
          if (g.row_stats) {
            float x[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) x[jj] = g.alpha * __uint_as_float(r[jj]);
            fold_row_stats(x, min(32, g.N - col0), rm, rs);
          }
          if (!row_on || col0 >= g.N) continue;
          if (g.vec && col0 + 32 <= g.N) {
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
              float4 v = make_float4(g.alpha * __uint_as_float(r[jj]), g.alpha * __uint_as_float(r[jj + 1]),
                                     g.alpha * __uint_as_float(r[jj + 2]), g.alpha * __uint_as_float(r[jj + 3]));
              float4* p = reinterpret_cast<float4*>(crow + col0 + jj);
              if (g.accumulate) {
                const float4 o = *p;
                v.x += o.x;
                v.y += o.y;
                v.z += o.z;
                v.w += o.w;
              }
              *p = v;
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              if (col0 + jj < g.N) {
                const float v = g.alpha * __uint_as_float(r[jj]);
                crow[col0 + jj] = g.accumulate ? crow[col0 + jj] + v : v;
              }
            }
          }
        }
        if (g.row_stats && row_on) g.row_stats[(int64_t)row * n_tiles + nt] = make_float2(rm, rs);
      }
      // this warp is done with accumulator buffer b: tell the MMA thread
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive_local(&tempty[b]);
        else mbar_arrive_remote_release(tempty_lead + 8u * (uint32_t)b);
      }
    }
    if (lane == 0) bulk_wait_all();
  }
  // both CTAs are done with the pair's TMEM (the peer's epilogue waited for
  // every MMA into it) before the pair releases it
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kTmemCols);
  }
}

sf_status make_map_c(CUtensorMap* map, float* C, int64_t M, int64_t N, int64_t ldc) {
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)(ldc * 4)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = tensor_map_encoder()(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, strides, box, estr,
                                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SF_ERR_CUDA, "cuTensorMapEncodeTiled (C) failed (%d)", (int)r);
  return SF_OK;
}

// bf16 operand map: a row-major [outer][ld] matrix read as boxes of 64
// inner elements (128 bytes, swizzled) by box_outer rows.  K-major operands
// have K inner (box_outer = their rows in a CTA), MN-major ones MN inner
// (box_outer = 64 K rows).
sf_status make_map(CUtensorMap* map, const void* base, int64_t inner, int64_t outer, int64_t ld, int box_outer) {
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = tensor_map_encoder()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SF_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SF_OK;
}

// An MN-major operand [K][ld] (MN inner, a multiple of 64) viewed in 3D as
// {64 MN, K, MN / 64 blocks} with the blocks 128 bytes apart, so one box
// {64, 64, 2} brings the 128 MN rows a CTA needs for a K slab (two 64 x 64
// swizzled blocks, one after the other) in one copy.  Every address of the
// view lies inside the matrix; false if the driver does not take the map.
bool make_map_mn3d(CUtensorMap* map, const void* base, int64_t mn, int64_t K, int64_t ld) {
  if (mn % 64) return false;
  cuuint64_t dims[3] = {64u, (cuuint64_t)K, (cuuint64_t)(mn / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), 128u};
  cuuint32_t box[3] = {64u, (cuuint32_t)kBK, 2u};
  cuuint32_t estr[3] = {1, 1, 1};
  return tensor_map_encoder()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of two GEMM CTAs that fit on the device at once (cached per
// device): the persistent grid's size.
sf_status resident_pairs(cudaLaunchConfig_t* cfg, int* out) {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  SF_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it == cache.end()) {
    int n = 0;
    cfg->gridDim = dim3((unsigned)(kPair * std::max(1, sm_count() / kPair)));
    SF_CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, k_tc_gemm, cfg), "cudaOccupancyMaxActiveClusters (k_tc_gemm)");
    if (n < 1) return fail(SF_ERR_UNSUPPORTED, "no cluster of two GEMM CTAs fits on this device");
    it = cache.emplace(dev, n).first;
  }
  *out = it->second;
  return SF_OK;
}

}  // namespace

// C = alpha A B^T (+ C); shared with the cross-entropy unit.
sf_status tc_gemm(const void* A, bool a_mn, const void* B, bool b_mn, float* C, int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc, float alpha, bool accumulate, cudaStream_t s,
                  float2* row_stats) {
  if (!A || !B || !C) return fail(SF_ERR_INVALID, "A, B or C is NULL");
  if (M < 1 || N < 1 || K < 1) return fail(SF_ERR_INVALID, "M, N, K must be >= 1");
  if (M > INT32_MAX - 2 * kPair * kBM || N > INT32_MAX - kBN || K > INT32_MAX - kBK)
    return fail(SF_ERR_UNSUPPORTED, "M, N, K must be below 2^31");
  if (lda < (a_mn ? M : K) || ldb < (b_mn ? N : K) || ldc < N)
    return fail(SF_ERR_INVALID, "leading dimensions must be >= the stored rows' length (lda: K or M, ldb: K or N; "
                                "ldc: N)");
  if ((lda * 2) % 16 || (ldb * 2) % 16 || (reinterpret_cast<uintptr_t>(A) % 16) ||
      (reinterpret_cast<uintptr_t>(B) % 16))
    return fail(SF_ERR_UNSUPPORTED, "A and B need 16-byte aligned bases and rows (lda, ldb multiples of 8)");
  if (!tensor_map_encoder()) return fail(SF_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available");
  // the tensor maps below may only address this device's own memory
  if (!on_current_device(A) || !on_current_device(B) || !on_current_device(C))
    return fail(SF_ERR_INVALID, "A, B and C must be device memory of the current device");
  CUtensorMap ma, mb;
  int a_form = 0, b_form = 0;      // 0 K-major, 1 MN-major in 2D boxes, 2 MN-major in 3D boxes
  if (a_mn) {
    a_form = make_map_mn3d(&ma, A, M, K, lda) ? 2 : 1;
    if (a_form == 1) SF_TRY(make_map(&ma, A, M, K, lda, kBK));
  } else {
    SF_TRY(make_map(&ma, A, K, M, lda, kBM));
  }
  if (b_mn) {
    b_form = make_map_mn3d(&mb, B, N, K, ldb) ? 2 : 1;
    if (b_form == 1) SF_TRY(make_map(&mb, B, N, K, ldb, kBK));
  } else {
    SF_TRY(make_map(&mb, B, K, N, ldb, kBRows));
  }
  TcGemmArgs g;
  g.C = C;
  g.ldc = ldc;
  g.M = (int32_t)M;
  g.N = (int32_t)N;
  g.K = (int32_t)K;
  g.alpha = alpha;
  g.accumulate = accumulate ? 1 : 0;
  g.vec = (ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(C) % 16 == 0) ? 1 : 0;
  g.tma = g.vec;
  g.n_fast = M > N ? 1 : 0;
  g.a_mn = a_form;
  g.b_mn = b_form;
  g.row_stats = row_stats;
  CUtensorMap mc = ma;       // unused unless g.tma
  if (g.tma) SF_TRY(make_map_c(&mc, C, M, N, ldc));
  SF_TRY(allow_dynamic_smem(reinterpret_cast<const void*>(&k_tc_gemm), kGemmSmem));
  const int64_t tiles = ((M + kPair * kBM - 1) / (kPair * kBM)) * ((N + kBN - 1) / kBN);
  if (tiles > INT32_MAX) return fail(SF_ERR_UNSUPPORTED, "too many tiles");
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int pairs = 0;
  SF_TRY(resident_pairs(&cfg, &pairs));
  cfg.gridDim = dim3((unsigned)(kPair * std::min<int64_t>(tiles, pairs)));
  SF_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_tc_gemm, ma, mb, mc, g), "launch k_tc_gemm");
  return SF_OK;
}

int read_and_clear_device_error_gemm() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof z);
  return v;
}

}  // namespace sf

extern "C" {

sf_status sf_gemm_abt_bf16(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                           int64_t ldb, int64_t ldc, float alpha, int accumulate, void* stream) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("sf_gemm_abt_bf16");
  return sf::tc_gemm(A, false, B, false, C, M, N, K, lda, ldb, ldc, alpha, accumulate != 0, sf::as_stream(stream),
                     nullptr);
}

sf_status sf_gemm_bf16(const void* A, int a_layout, const void* B, int b_layout, float* C, int64_t M, int64_t N,
                       int64_t K, int64_t lda, int64_t ldb, int64_t ldc, float alpha, int accumulate, void* stream) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("sf_gemm_bf16");
  if ((a_layout != 0 && a_layout != 1) || (b_layout != 0 && b_layout != 1))
    return sf::fail(SF_ERR_INVALID, "a_layout and b_layout must be 0 (K-major) or 1 (MN-major)");
  return sf::tc_gemm(A, a_layout == 1, B, b_layout == 1, C, M, N, K, lda, ldb, ldc, alpha, accumulate != 0,
                     sf::as_stream(stream), nullptr);
}

}  // extern "C"

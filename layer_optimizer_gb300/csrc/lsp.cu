// Learned-sparse-projector path: projector bookkeeping, compress
// S = P^T G Q, decompress-apply W -= P dS Q^T.
//
// "Practical offloading for fine-tuning LLM on commodity GPU via learned
// sparse projectors" (LSP-Offload; abstract and method section) compresses
// the gradient with sparse projectors holding a fixed number k of nonzeros
// per row, updates in the d x d compressed space and decompresses the step
// back.  The pages give no kernel; everything below is designed for sm_103a.
//
// Why no tensor cores: P and Q are k/d dense (8/512 = 1.6 %); a dense
// product would do d/k = 64x the useful multiply-adds.  The work is a
// gather: every G element meets k projector entries, 2 multiply-adds per
// G byte (fp32 G, k = 8).  The kernels stream the big matrix once through
// shared memory and keep the lanes of a warp on its contiguous dimension,
// so every gathered shared-memory access is conflict-free and every
// projector entry is a warp-uniform broadcast.
//
// Compress, two gathers (R-first):
//   stage 1  R^T = (P^T G)^T      k_gather_t over G, A = P      (n x d)
//   stage 2  S   = (Q^T R^T)^T    k_rowgather over R^T, A = Q   (d x d)
//            (R^T is small and still in L2: read straight from there;
//            k_gather_t when its rows are not 16-byte multiples)
// k_gather_t(A, B) writes Y^T = (A^T B)^T: a CTA owns 128 columns of B and
// 4 x warps outputs a (columns of A; 32 warps, 128 outputs for d >= 128);
// B streams through shared memory in windows of 128 rows by TMA
// (cp.async.bulk.tensor); the CTAs that share a column block each load the
// window themselves (the repeats come from L2).  A's entries come from a
// window-major column list (entries of window w and column a, rows
// ascending, with a prefix table), so a warp finds its (window, a) entries
// with a few broadcast loads.  Row splits (for grid size) write partial
// outputs that one reduction sums in split order; grids past whole waves
// split only the column blocks left over after the whole waves.  The CTAs
// that read the same windows (one per output range) are dispatched next to
// each other, so each tile comes from DRAM once.  A layer's matrices can go
// through one launch per stage (k_gather_t_multi, k_rowgather_multi), every
// tile computed as in its own launch.
//
// Measured on GB300 for one 4096 x 4096 fp32 G (stage 1, 134 M multiply-
// adds): this kernel 46 us; k_rowgather reading G's rows straight from L2
// instead 61 us (same bits; latency-bound at a quarter of L2's throughput);
// the shared-memory pipe runs about 60 % busy and the warps wait mostly on
// shared-memory loads and tile arrival.  Tensor memory (tcgen05.ld) reads
// faster than shared memory only four columns per lane at a time, and a
// warp reaches only its quarter of TMEM's lanes, so holding a window there
// would split every output's accumulators over the quarters.
//
// Decompress:
//   V = dS Q^T (d x n)          k_transpose_dd + k_v_rows: row gathers of
//                               dS^T (k = 8); k_v: dS^T block resident in
//                               shared memory, Q rows as warp-uniform entries
//   W[i, :] -= sum_l P[i,a_l] V[a_l, :]   k_apply: a 64-column block of V
//                               resident in shared memory, W read and
//                               written once, coalesced.
// Nothing uses atomics on floating-point data: every sum has a fixed order,
// so results are bitwise deterministic.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>
#include <new>
#include <vector>

#include "common.h"
#include "lsp_internal.cuh"
#include "ptx.cuh"

namespace sf {
namespace {

constexpr int kWinRows = 128;       // rows of A (and of B) per window
constexpr int kColsPerCta = 128;    // B columns per gather CTA (4 per lane)
constexpr int kGatherOut = 4;       // outputs (columns of A) per gather warp
constexpr int kMaxStages = 4;       // TMA ring depth of the gather kernel (at most)
constexpr int kTargetCtas = 148;    // grid size aimed at (about one CTA per SM)
constexpr int kWaveCtas = 152;      // gather CTAs of one wave on a GB300 (one per SM)
constexpr int kApplyCols = 64;      // W columns per apply CTA (2 per lane)
constexpr int kVRows = 64;          // a rows per V CTA (2 per lane)
constexpr int kMaxFastD = 512;      // shared-memory tiles of k_v / k_apply hold d <= 512

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }

}  // namespace
}  // namespace sf


namespace sf {
namespace {

// ----------------------------------------------------------------------------
// Bookkeeping kernels (run once per projector)
// ----------------------------------------------------------------------------

// Per-window histogram of column ids.  Out-of-range ids are dropped and flagged.
__global__ void k_window_hist(const int32_t* __restrict__ idx, int64_t rows, int k, int d, int dp,
                              int32_t* __restrict__ wcnt, int32_t* __restrict__ err) {
  extern __shared__ int32_t sh[];
  const int w = blockIdx.x;
  for (int c = threadIdx.x; c < dp; c += blockDim.x) sh[c] = 0;
  __syncthreads();
  const int64_t e0 = (int64_t)w * kWinRows * k;
  const int64_t e1 = min(rows, (int64_t)(w + 1) * kWinRows) * k;
  for (int64_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
    const int c = idx[e];
    if (c >= 0 && c < d) atomicAdd(&sh[c], 1);
    else atomicOr(err, kDevErrIndex);
  }
  __syncthreads();
  for (int c = threadIdx.x; c < dp; c += blockDim.x) wcnt[(int64_t)w * dp + c] = sh[c];
}

// Per column: exclusive offsets over windows, and the column total.
__global__ void k_column_offsets(const int32_t* __restrict__ wcnt, int n_win, int d, int dp,
                                 int32_t* __restrict__ csc_off, int32_t* __restrict__ totals) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  int32_t off = 0;
  for (int w = 0; w < n_win; ++w) {
    csc_off[(int64_t)w * dp + c] = off;
    off += wcnt[(int64_t)w * dp + c];
  }
  totals[c] = off;
}

// Single-block exclusive scan: out[i] = sum(in[0..i)), out[n] = total.
__global__ void k_scan_exclusive(const int32_t* __restrict__ in, int64_t n, int32_t* __restrict__ out) {
  __shared__ int32_t part[1024];
  const int t = threadIdx.x, T = blockDim.x;
  const int64_t per = (n + T - 1) / T;
  const int64_t b = min(n, per * t), e = min(n, b + per);
  int32_t s = 0;
  for (int64_t i = b; i < e; ++i) s += in[i];
  part[t] = s;
  __syncthreads();
  if (t == 0) {
    int32_t run = 0;
    for (int i = 0; i < T; ++i) {
      const int32_t v = part[i];
      part[i] = run;
      run += v;
    }
    out[n] = run;
  }
  __syncthreads();
  int32_t run = part[t];
  for (int64_t i = b; i < e; ++i) {
    const int32_t v = in[i];
    out[i] = run;
    run += v;
  }
}

// One warp per window: stable placement of the window's entries into the
// column lists (CSC) and the window-major lists.  Within a window the
// entries are visited in ELL order (row-major), so rows ascend inside every
// column; equal ids of one warp step are ranked by lane.
__global__ void k_place(const int32_t* __restrict__ idx, const float* __restrict__ val, int64_t rows, int k,
                        int d, int dp, int n_win, const int32_t* __restrict__ wptr,
                        const int32_t* __restrict__ csc_off, const int32_t* __restrict__ col_ptr,
                        int2* __restrict__ went, int32_t* __restrict__ row_idx, float* __restrict__ csc_val,
                        int32_t* __restrict__ ell2csc, int32_t* __restrict__ ell2went) {
  extern __shared__ int32_t cnt_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * (blockDim.x >> 5) + warp;
  int32_t* cnt = cnt_all + warp * dp;
  for (int c = lane; c < dp; c += 32) cnt[c] = 0;
  __syncwarp();
  if (w >= n_win) return;
  const int64_t e0 = (int64_t)w * kWinRows * k;
  const int64_t e1 = min(rows, (int64_t)(w + 1) * kWinRows) * k;
  const unsigned lt = (1u << lane) - 1u;
  for (int64_t base_e = e0; base_e < e1; base_e += 32) {
    const int64_t e = base_e + lane;
    int c = -1;
    if (e < e1) {
      c = idx[e];
      if (c < 0 || c >= d) c = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    const int rank = __popc(peers & lt);
    int32_t base = 0;
    if (c >= 0) base = cnt[c];
    __syncwarp();
    if (c >= 0 && rank == __popc(peers) - 1) cnt[c] = base + __popc(peers);
    __syncwarp();
    if (c >= 0) {
      const int32_t row = (int32_t)(e / k);
      const float v = val[e];
      const int32_t pw = wptr[(int64_t)w * dp + c] + base + rank;
      went[pw] = make_int2(row, __float_as_int(v));
      const int32_t pc = col_ptr[c] + csc_off[(int64_t)w * dp + c] + base + rank;
      row_idx[pc] = row;
      csc_val[pc] = v;
      ell2csc[e] = pc;
      ell2went[e] = pw;
    }
  }
}

// Column order by (nnz bucket, column id); bucket 0 = empty, else ceil(log2 nnz) + 1.
// One block, a thread per column (d <= 1024): each column's key is
// (bucket, id), unique, and its place in the order is the number of smaller
// keys, counted over all columns from shared memory.
__global__ void k_bucket_perm(const int32_t* __restrict__ col_ptr, int d, int32_t* __restrict__ perm) {
  __shared__ int32_t key[1024];
  const int c = threadIdx.x;
  int my = INT32_MAX;
  if (c < d) {
    const int nnz = col_ptr[c + 1] - col_ptr[c];
    int bucket = 0;
    if (nnz > 0) {
      int b = 0;
      while ((1 << b) < nnz) ++b;
      bucket = b + 1;
    }
    my = bucket * 1024 + c;
  }
  key[c] = my;
  __syncthreads();
  if (c < d) {
    int rank = 0;
    for (int i = 0; i < d; ++i) rank += key[i] < my ? 1 : 0;
    perm[rank] = c;
  }
}

// Validation: ids in range and no id repeated inside a row.
__global__ void k_validate_rows(const int32_t* __restrict__ idx, int64_t rows, int k, int d,
                                int32_t* __restrict__ err) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  const int32_t* p = idx + r * k;
  for (int a = 0; a < k; ++a) {
    const int ca = p[a];
    if (ca < 0 || ca >= d) {
      atomicOr(err, kDevErrIndex);
      return;
    }
    for (int b = 0; b < a; ++b)
      if (p[b] == ca) {
        atomicOr(err, 4);
        return;
      }
  }
}

// Copy of the ELL with out-of-range entries neutralised (id 0, value 0).
__global__ void k_copy_ell(const int32_t* __restrict__ idx, const float* __restrict__ val, int64_t n, int d,
                           int32_t* __restrict__ oidx, float* __restrict__ oval) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int c = idx[e];
    const bool ok = c >= 0 && c < d;
    oidx[e] = ok ? c : 0;
    oval[e] = ok ? val[e] : 0.0f;
  }
}

// Per (a-range, window): the slice of the window-major list that one gather
// CTA needs, as a 16-byte aligned (first entry, byte count) pair for a bulk copy.
__global__ void k_gdesc(const int32_t* __restrict__ wptr, int n_win, int dp, int a_rng, int n_ar,
                        int2* __restrict__ gdesc, int32_t* __restrict__ max_bytes) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)n_win * n_ar) return;
  const int w = (int)(t % n_win), ar = (int)(t / n_win);
  const int lo = ar * a_rng, hi = min(lo + a_rng, dp);
  const int32_t e0 = wptr[(int64_t)w * dp + lo], e1 = wptr[(int64_t)w * dp + hi];
  const int32_t e0a = e0 & ~1;
  const int32_t bytes = ((e1 - e0a) * 8 + 15) / 16 * 16;
  gdesc[t] = make_int2(e0a, bytes);
  atomicMax(max_bytes, bytes);
}

// ----------------------------------------------------------------------------
// Gather kernel: Y^T = (A^T B)^T with TMA-staged windows of B
// ----------------------------------------------------------------------------

struct GatherArgs {
  const int32_t* wptr;
  const int2* went;
  const int2* gdesc;
  float* yt;               // [ncols][d]: Y^T (or split 0's partial, see direct0)
  float* part;             // partial outputs of row splits (see direct0)
  int64_t split_stride;    // elements between split outputs
  int32_t direct0;         // 1: split 0 writes Y^T and split z >= 1 partial z - 1; 0: split z writes partial z
  int32_t out_c0;          // first column a partial holds
  int32_t main_tiles;      // > 0: 1D grid, whole tiles then the split tail (see k_gather_t)
  int32_t cb_main;         // column blocks done whole (1D grid)
  int32_t n_cb, n_ar;      // column blocks, output ranges (1D grid)
  int32_t tail_wps;        // windows per split of the tail (1D grid)
  int32_t ncols;           // columns of B
  int32_t d, dp;           // columns of A (outputs a)
  int32_t n_win;           // windows of A / B rows
  int32_t win_per_split;
  int32_t cbx;             // B tile row width in elements (<= 128)
  int32_t stage_tx;        // bytes of one full window tile
  int32_t wsl_off;         // offset of the staged prefix-table slice inside a stage
  int32_t wbytes;          // its bytes (8 x warps + 1 ints, padded to 16)
  int32_t ent_off;         // offset of the staged entry slice inside a stage
  int32_t stage_stride;    // bytes between stages in shared memory
  int32_t vec_out;         // output rows are 16-byte aligned (d % 4 == 0, aligned base)
  int32_t stages;          // depth of the TMA ring
};

// 4 consecutive B elements of a tile row as fp32 (bf16 widened exactly).
template <typename TB>
__device__ __forceinline__ float4 tile_load(uint32_t addr) {
  if constexpr (sizeof(TB) == 4) {
    return lds_f4(addr);
  } else {
    const uint2 u = lds_u2(addr);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
  }
}

// The same 4 elements as two packed fp32 pairs (first pair in .x).
template <typename TB>
__device__ __forceinline__ ulonglong2 tile_load2(uint32_t addr) {
  if constexpr (sizeof(TB) == 4) {
    return lds_u64x2(addr);
  } else {
    const uint2 u = lds_u2(addr);
    return make_ulonglong2(pack_f2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u)),
                           pack_f2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u)));
  }
}

// One CTA: kGatherOut outputs per warp, as many warps as the projector's
// output range needs (32 for d >= 128).  There is no producer warp: lane 0
// of the last warp issues the copies of a stage once every warp has released
// it, before it computes its own share of the next window, so all warps of
// the CTA gather (twice the warps per SM of a dedicated producer layout,
// which keeps the shared-memory loads' latency hidden).
//
// The tile of a CTA: column block cb, output range ar, row split z of wps
// windows.  On a 1D grid (A.main_tiles > 0) blocks [0, main_tiles) take the
// first cb_main column blocks whole (whole waves of the GPU) and the rest
// split the windows of the remaining column blocks, so the last wave is not
// left with a few whole tiles; otherwise the blocks walk (output range,
// column block, split).  Either way the output range varies fastest, so the
// CTAs that read the same windows of B are dispatched together and each
// tile comes from DRAM once, whatever wave they fall in.
struct GatherTile {
  int cb, ar, z, wps;
};

__device__ __forceinline__ GatherTile tile_of_block(const GatherArgs& A, int b) {
  GatherTile t;
  if (A.main_tiles > 0) {
    if (b < A.main_tiles) {
      t.ar = b % A.n_ar;
      t.cb = b / A.n_ar;
      t.z = 0;
      t.wps = A.n_win;
    } else {
      const int r = b - A.main_tiles, tail_splits = (A.n_win + A.tail_wps - 1) / A.tail_wps;
      t.ar = r % A.n_ar;
      t.z = (r / A.n_ar) % tail_splits;
      t.cb = A.cb_main + r / (A.n_ar * tail_splits);
      t.wps = A.tail_wps;
    }
  } else {
    t.ar = b % A.n_ar;
    t.cb = (b / A.n_ar) % A.n_cb;
    t.z = b / (A.n_ar * A.n_cb);
    t.wps = A.win_per_split;
  }
  return t;
}

template <typename TB>
__device__ __forceinline__ void gather_tile(const CUtensorMap* map, const GatherArgs& A, const GatherTile tile) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // round up to 1024 with arithmetic on the __shared__ array itself, so the
  // compiler keeps the shared address space (plain LDS, not generic loads)
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = A.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * A.stage_stride);
  uint64_t* empty = full + kMaxStages;
  int32_t* hdr = reinterpret_cast<int32_t*>(empty + kMaxStages);   // first staged entry of each stage
  int32_t* flags = hdr + kMaxStages;                                // [0] issued, [1] failed

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int cb = tile.cb, ar = tile.ar, z = tile.z, wps = tile.wps;
  const int c0 = cb * kColsPerCta;
  const int a_cta = ar * kGatherOut * nwarps;
  const int w_begin = z * wps;
  const int w_end = min(A.n_win, w_begin + wps);
  const int nw = max(0, w_end - w_begin);
  const bool producer = warp == nwarps - 1 && lane == 0;

  if (threadIdx.x == 0) {
    prefetch_tensormap(map);
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nwarps);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init_cluster();
  }
  __syncthreads();
  griddep_launch_dependents();

  // one stage = the B tile of a window, this CTA's slice of the prefix
  // table and its entry slice
  const int2* gd_row = A.gdesc + (int64_t)ar * A.n_win;
  auto issue = [&](int it) {
    const int s = it % S;
    const int w = w_begin + it;
    const int2 gd = gd_row[w];
    unsigned char* st = smem + (size_t)s * A.stage_stride;
    hdr[s] = gd.x;
    mbar_arrive_expect_tx(&full[s], (uint32_t)(A.stage_tx + A.wbytes + gd.y));
    tma_load_2d(st, map, &full[s], c0, w * kWinRows);
    bulk_load(st + A.wsl_off, A.wptr + (int64_t)w * A.dp + a_cta, (uint32_t)A.wbytes, &full[s]);
    if (gd.y > 0) bulk_load(st + A.ent_off, A.went + gd.x, (uint32_t)gd.y, &full[s]);
  };
  int issued = 0;
  if (producer) {
    griddep_wait();            // B may be the previous kernel's output
    for (; issued < min(S, nw); ++issued) issue(issued);
    flags[0] = issued;
  }

  const int a0 = a_cta + kGatherOut * warp;
  const bool lane_on = 4 * lane < A.cbx;
  const bool warp_on = a0 < A.dp;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t row_bytes = (uint32_t)A.cbx * (uint32_t)sizeof(TB);
  const uint32_t lane_off = 4u * (uint32_t)lane * (uint32_t)sizeof(TB);
  // the lane's 4 columns of each output as two packed fp32 pairs
  uint64_t acc[kGatherOut][2];
#pragma unroll
  for (int sl = 0; sl < kGatherOut; ++sl) acc[sl][0] = acc[sl][1] = 0ull;
  bool failed = false;
  int s = 0;
  uint32_t pass = 0;
  const uint32_t full_a = smem_u32(full);
  for (int it = 0; it < nw; ++it) {
    // refill the stage of the previous window for window it - 1 + S once
    // every warp has released it (this warp released it last iteration)
    if (producer && it >= 1 && issued < nw && !failed) {
      const int prev = it - 1;
      if (!mbar_wait_u32(smem_u32(&empty[prev % S]), (uint32_t)(prev / S) & 1u)) {
        failed = true;
        flags[1] = 1;
      } else {
        issue(issued++);
        flags[0] = issued;
      }
    }
    if (failed || !mbar_wait_u32(full_a + 8u * (uint32_t)s, pass)) {
      failed = true;
      flags[1] = 1;
      break;
    }
    const int w = w_begin + it;
    if (warp_on && lane_on) {
      // 32-bit shared addresses: entry i of the stage at ent + 8 i; row r of
      // the tile, this lane's 4 columns, at row_adj + r * row_bytes
      const uint32_t tile = smem_base + (uint32_t)s * (uint32_t)A.stage_stride;
      const uint32_t bp = tile + (uint32_t)A.wsl_off + 4u * kGatherOut * (uint32_t)warp;
      int bnd[kGatherOut + 1];
#pragma unroll
      for (int q = 0; q <= kGatherOut; ++q) bnd[q] = (int)lds_u32(bp + 4u * q);
      const int32_t e_base = hdr[s];
      const uint32_t ent = tile + (uint32_t)A.ent_off - 8u * (uint32_t)e_base;
      const uint32_t row_adj = tile + lane_off - (uint32_t)(w * kWinRows) * row_bytes;
#pragma unroll
      for (int sl = 0; sl < kGatherOut; ++sl) {
        uint32_t ea = ent + 8u * (uint32_t)bnd[sl];
        const uint32_t ee = ent + 8u * (uint32_t)bnd[sl + 1];
        uint64_t a01 = acc[sl][0], a23 = acc[sl][1];
        // two entries per step: both entry loads, then both tile loads, in flight together
        for (; ea + 8u < ee; ea += 16u) {
          const int2 en0 = lds_i2(ea);
          const int2 en1 = lds_i2(ea + 8u);
          const ulonglong2 x0 = tile_load2<TB>(row_adj + (uint32_t)en0.x * row_bytes);
          const ulonglong2 x1 = tile_load2<TB>(row_adj + (uint32_t)en1.x * row_bytes);
          const float v0 = __int_as_float(en0.y), v1 = __int_as_float(en1.y);
          const uint64_t vv0 = pack_f2(v0, v0), vv1 = pack_f2(v1, v1);
          ffma2(a01, x0.x, vv0);
          ffma2(a23, x0.y, vv0);
          ffma2(a01, x1.x, vv1);
          ffma2(a23, x1.y, vv1);
        }
        if (ea < ee) {
          const int2 en = lds_i2(ea);
          const ulonglong2 x = tile_load2<TB>(row_adj + (uint32_t)en.x * row_bytes);
          const float v = __int_as_float(en.y);
          const uint64_t vv = pack_f2(v, v);
          ffma2(a01, x.x, vv);
          ffma2(a23, x.y, vv);
        }
        acc[sl][0] = a01;
        acc[sl][1] = a23;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_local(&empty[s]);
    if (++s == S) {
      s = 0;
      pass ^= 1u;
    }
  }

  // Y^T[col][a] for the lane's 4 columns and the warp's outputs.
  if (warp_on && lane_on && !failed) {
    float res[kGatherOut][4];
#pragma unroll
    for (int sl = 0; sl < kGatherOut; ++sl) {
      const float2 p01 = unpack_f2(acc[sl][0]), p23 = unpack_f2(acc[sl][1]);
      res[sl][0] = p01.x;
      res[sl][1] = p01.y;
      res[sl][2] = p23.x;
      res[sl][3] = p23.y;
    }
    const bool to_yt = z == 0 && A.direct0;
    float* out = to_yt ? A.yt : A.part + (int64_t)(z - A.direct0) * A.split_stride;
    const int oc0 = to_yt ? 0 : A.out_c0;
    const bool vec = A.vec_out && (a0 + kGatherOut <= A.d);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = c0 + 4 * lane + j;
      if (col >= A.ncols) continue;
      float* o = out + (int64_t)(col - oc0) * A.d + a0;
      if (vec) {
        *reinterpret_cast<float4*>(o) = make_float4(res[0][j], res[1][j], res[2][j], res[3][j]);
      } else {
#pragma unroll
        for (int sl = 0; sl < kGatherOut; ++sl)
          if (a0 + sl < A.d) o[sl] = res[sl][j];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && flags[1]) {
    // a wait ran out: let this CTA's copies still in flight land (bounded)
    const int n_issued = flags[0];
    for (int j = max(0, n_issued - S); j < n_issued; ++j) mbar_wait(&full[j % S], (uint32_t)(j / S) & 1u);
  }
}

template <typename TB>
__global__ void __launch_bounds__(1024, 1) k_gather_t(const __grid_constant__ CUtensorMap map,
                                                      const __grid_constant__ GatherArgs A) {
  const GatherTile t = A.main_tiles > 0 ? tile_of_block(A, blockIdx.x)
                                        : GatherTile{(int)blockIdx.x, (int)blockIdx.y, (int)blockIdx.z, A.win_per_split};
  gather_tile<TB>(&map, A, t);
}

// Several gathers of the same block shape in one launch (the matrices of a
// layer): block b belongs to the gather whose [block_begin, block_end) holds
// it and runs that gather's tile of the same index, so every tile is
// computed exactly as in its own launch.
constexpr int kMaxLayerMats = 8;
struct MultiGatherArgs {
  CUtensorMap map[kMaxLayerMats];
  GatherArgs a[kMaxLayerMats];
  int32_t block_end[kMaxLayerMats];
  int32_t count;
};

template <typename TB>
__global__ void __launch_bounds__(1024, 1) k_gather_t_multi(const __grid_constant__ MultiGatherArgs M) {
  int i = 0;
  while (i + 1 < M.count && (int)blockIdx.x >= M.block_end[i]) ++i;
  const int b = (int)blockIdx.x - (i > 0 ? M.block_end[i - 1] : 0);
  gather_tile<TB>(&M.map[i], M.a[i], tile_of_block(M.a[i], b));
}

// Generic gather for shapes the TMA path cannot take: one thread per output.
template <typename TB>
__global__ void k_gather_generic(const TB* __restrict__ B, int64_t ldb, int64_t ncols, int d,
                                 const int32_t* __restrict__ col_ptr, const int32_t* __restrict__ row_idx,
                                 const float* __restrict__ csc_val, float* __restrict__ yt) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= ncols * d) return;
  const int a = (int)(t % d);
  const int64_t col = t / d;
  float acc = 0.0f;
  for (int e = col_ptr[a]; e < col_ptr[a + 1]; ++e) {
    float b;
    if constexpr (sizeof(TB) == 4) b = B[(int64_t)row_idx[e] * ldb + col];
    else b = __bfloat162float(B[(int64_t)row_idx[e] * ldb + col]);
    acc = fmaf(csc_val[e], b, acc);
  }
  yt[col * d + a] = acc;
}

// Second compress stage when the dense operand is small and L2-resident
// (B = R^T, n x d fp32, just written by stage 1):
//   yt[c][a] = sum over the entries (j, q) of column a of A (rows ascending)
//              of q * B[j][c]
// One warp per output column a and 128-column slice of B: the warp fetches
// 32 entries at a time (one per lane), broadcasts them in order, and each
// lane reads 4 consecutive columns of row j (16-byte loads, sixteen rows
// in flight), so B is read straight from L2 with no staging and no split
// partials.  The CTA's 8 outputs are transposed through shared memory so
// yt is written as 32-byte row segments.  Needs B 16-byte aligned with
// ldb and ncols multiples of 4 (every 16-byte load inside a row).
constexpr int kRgWarps = 8, kRgCols = 128, kRgUnroll = 16;
struct RowGatherArgs {
  const float* B;
  int64_t ldb;
  int ncols;
  const int32_t* col_ptr;
  const int32_t* row_idx;
  const float* csc_val;
  int d;
  float* yt;
};

__device__ __forceinline__ void rowgather_block(const float* __restrict__ B, int64_t ldb, int ncols,
                                                const int32_t* __restrict__ col_ptr,
                                                const int32_t* __restrict__ row_idx,
                                                const float* __restrict__ csc_val, int d, float* __restrict__ yt,
                                                int bx, int by) {
  __shared__ float tile[kRgWarps][kRgCols + 4];
  griddep_launch_dependents();
  griddep_wait();                // B is the previous kernel's output
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a0 = bx * kRgWarps, a = a0 + warp;
  const int c0 = by * kRgCols, c = c0 + 4 * lane;
  const bool col_on = c < ncols;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (a < d) {
    const int e0 = col_ptr[a], e1 = col_ptr[a + 1];
    for (int eb = e0; eb < e1; eb += 32) {
      int jl = 0;
      float ql = 0.0f;
      if (eb + lane < e1) {
        jl = row_idx[eb + lane];
        ql = csc_val[eb + lane];
      }
      const int cnt = min(32, e1 - eb);
      int t = 0;
      for (; t + kRgUnroll <= cnt; t += kRgUnroll) {
        float4 x[kRgUnroll];
        float q[kRgUnroll];
#pragma unroll
        for (int u = 0; u < kRgUnroll; ++u) {
          const int j = __shfl_sync(0xffffffffu, jl, t + u);
          q[u] = __shfl_sync(0xffffffffu, ql, t + u);
          x[u] = col_on ? *reinterpret_cast<const float4*>(B + (int64_t)j * ldb + c)
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < kRgUnroll; ++u) {
          acc.x = fmaf(q[u], x[u].x, acc.x);
          acc.y = fmaf(q[u], x[u].y, acc.y);
          acc.z = fmaf(q[u], x[u].z, acc.z);
          acc.w = fmaf(q[u], x[u].w, acc.w);
        }
      }
      for (; t < cnt; ++t) {
        const int j = __shfl_sync(0xffffffffu, jl, t);
        const float q = __shfl_sync(0xffffffffu, ql, t);
        const float4 x = col_on ? *reinterpret_cast<const float4*>(B + (int64_t)j * ldb + c)
                                : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        acc.x = fmaf(q, x.x, acc.x);
        acc.y = fmaf(q, x.y, acc.y);
        acc.z = fmaf(q, x.z, acc.z);
        acc.w = fmaf(q, x.w, acc.w);
      }
    }
  }
  tile[warp][4 * lane] = acc.x;
  tile[warp][4 * lane + 1] = acc.y;
  tile[warp][4 * lane + 2] = acc.z;
  tile[warp][4 * lane + 3] = acc.w;
  __syncthreads();
  for (int idx = threadIdx.x; idx < kRgCols * kRgWarps; idx += blockDim.x) {
    const int cc = idx / kRgWarps, w = idx % kRgWarps;
    if (c0 + cc < ncols && a0 + w < d) yt[(int64_t)(c0 + cc) * d + a0 + w] = tile[w][cc];
  }
}

__global__ void __launch_bounds__(32 * kRgWarps, 2) k_rowgather(const float* __restrict__ B, int64_t ldb, int ncols,
                                                             const int32_t* __restrict__ col_ptr,
                                                             const int32_t* __restrict__ row_idx,
                                                             const float* __restrict__ csc_val, int d,
                                                             float* __restrict__ yt) {
  rowgather_block(B, ldb, ncols, col_ptr, row_idx, csc_val, d, yt, blockIdx.x, blockIdx.y);
}

// The second stage of several matrices in one launch: block b belongs to
// the matrix whose [block_begin, block_end) holds it and is that matrix's
// block (b % gx, b / gx) of its own grid.
struct MultiRowGatherArgs {
  RowGatherArgs a[kMaxLayerMats];
  int32_t gx[kMaxLayerMats];
  int32_t block_end[kMaxLayerMats];
  int32_t count;
};

__global__ void __launch_bounds__(32 * kRgWarps, 2) k_rowgather_multi(const __grid_constant__ MultiRowGatherArgs M) {
  int i = 0;
  while (i + 1 < M.count && (int)blockIdx.x >= M.block_end[i]) ++i;
  const int b = (int)blockIdx.x - (i > 0 ? M.block_end[i - 1] : 0);
  const RowGatherArgs& R = M.a[i];
  rowgather_block(R.B, R.ldb, R.ncols, R.col_ptr, R.row_idx, R.csc_val, R.d, R.yt, b % M.gx[i], b / M.gx[i]);
}

// out[e] = sum over splits s = 0, 1, ... of part[s][e], in that order.
__global__ void k_reduce_splits(const float* __restrict__ part, int splits, int64_t stride, int64_t n,
                                float* __restrict__ out) {
  griddep_launch_dependents();
  griddep_wait();
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    float s = 0.0f;
    for (int k = 0; k < splits; ++k) s += part[k * stride + e];
    out[e] = s;
  }
}

// out[e] = out[e] + part[0][e] + part[1][e] + ..., added in that order (the
// split tail of a 1D gather grid: split 0 wrote out itself).
__global__ void k_add_splits(const float* __restrict__ part, int n_part, int64_t stride, int64_t n,
                             float* __restrict__ out) {
  griddep_launch_dependents();
  griddep_wait();
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    float s = out[e];
    for (int k = 0; k < n_part; ++k) s += part[k * stride + e];
    out[e] = s;
  }
}

// ----------------------------------------------------------------------------
// Decompress kernels
// ----------------------------------------------------------------------------

constexpr int kVMaxK = 8;            // k_v keeps 8 x k entries per warp in shared memory
constexpr int kVWarps = 16;          // warps of a k_v CTA
constexpr int kVGroup = 8;           // V columns a warp computes at a time (one 32-byte sector per row)

__host__ __device__ __forceinline__ size_t v_ebuf_offset(int d) { return ((size_t)d * 65 * 4 + 15) / 16 * 16; }
__host__ __device__ __forceinline__ size_t v_smem_bytes(int d) {
  return v_ebuf_offset(d) + (size_t)kVWarps * kVGroup * kVMaxK * 8;
}

// V[a][j] = sum_l q_{j,l} dS[a][c_{j,l}] for a in a 64-row block and the
// CTA's range of columns j.  dS^T of the block sits in shared memory
// (st[c * 65 + aa], padded: the transposing fill and the lane-along-a reads
// are both conflict-free).  A warp takes 8 columns at a time: their 8 x k Q
// entries go through a small per-warp buffer and are read back as
// warp-uniform broadcasts; each lane keeps rows a0 + lane and a0 + lane + 32
// of the 8 columns in registers and writes them as two 32-byte row segments.
__global__ void __launch_bounds__(32 * kVWarps) k_v(const float* __restrict__ dS, int d,
                                                    const int32_t* __restrict__ qidx,
                                                    const float* __restrict__ qval, int k, int64_t n,
                                                    float* __restrict__ V, int64_t cols_per_cta) {
  extern __shared__ float st[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  unsigned char* sbytes = reinterpret_cast<unsigned char*>(st);
  int2* ebuf = reinterpret_cast<int2*>(sbytes + v_ebuf_offset(d)) + (size_t)warp * kVGroup * kVMaxK;
  const uint32_t ebuf_a = smem_u32(ebuf);
  const int a0 = blockIdx.x * kVRows;
  griddep_launch_dependents();
  griddep_wait();                // dS comes from the compressed step
  if ((d & 3) == 0 && (reinterpret_cast<uintptr_t>(dS) & 15) == 0) {
    // lanes along a (one dS row each), warps along 4-column groups: 16-byte
    // loads, 8 in flight per thread; the transposing stores hit 32 distinct banks
    const int c4n = d / 4;
    for (int half = 0; half < 2; ++half) {
      const int aa = lane + 32 * half;
      const int a = a0 + aa;
      for (int c4 = warp; c4 < c4n; c4 += 8 * nwarps) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int cc = c4 + u * nwarps;
          v[u] = (a < d && cc < c4n) ? *reinterpret_cast<const float4*>(dS + (int64_t)a * d + 4 * cc)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int cc = c4 + u * nwarps;
          if (cc < c4n) {
            st[(4 * cc + 0) * 65 + aa] = v[u].x;
            st[(4 * cc + 1) * 65 + aa] = v[u].y;
            st[(4 * cc + 2) * 65 + aa] = v[u].z;
            st[(4 * cc + 3) * 65 + aa] = v[u].w;
          }
        }
      }
    }
  } else {
    for (int aa = warp; aa < kVRows; aa += nwarps) {
      const int a = a0 + aa;
      for (int c = lane; c < d; c += 32) st[c * 65 + aa] = a < d ? dS[(int64_t)a * d + c] : 0.0f;
    }
  }
  __syncthreads();
  const uint32_t st_lo = smem_u32(st) + 4u * (uint32_t)lane;   // st[c * 65 + lane] at st_lo + 260 c
  const bool on_lo = a0 + lane < d, on_hi = a0 + lane + 32 < d;
  float* v_lo = V + (int64_t)(a0 + lane) * n;
  float* v_hi = V + (int64_t)(a0 + lane + 32) * n;
  const bool vec = (n & 3) == 0 && (reinterpret_cast<uintptr_t>(V) & 15) == 0;
  const int64_t j_begin = (int64_t)blockIdx.y * cols_per_cta;
  const int64_t j_end = imin64(n, j_begin + cols_per_cta);
  for (int64_t j0 = j_begin + kVGroup * warp; j0 < j_end; j0 += (int64_t)kVGroup * nwarps) {
    const int cols = (int)imin64(kVGroup, j_end - j0);
    const int ne = cols * k;
    __syncwarp();
    for (int e = lane; e < ne; e += 32)
      ebuf[e] = make_int2(qidx[j0 * k + e], __float_as_int(qval[j0 * k + e]));
    __syncwarp();
    float s_lo[kVGroup], s_hi[kVGroup];
#pragma unroll
    for (int u = 0; u < kVGroup; ++u) s_lo[u] = s_hi[u] = 0.0f;
    if (k == kVMaxK && cols == kVGroup) {
      // every load of the group is independent: fully unrolled
#pragma unroll
      for (int l = 0; l < kVMaxK; ++l) {
#pragma unroll
        for (int u = 0; u < kVGroup; ++u) {
          const int2 en = lds_i2(ebuf_a + 8u * (uint32_t)(u * kVMaxK + l));
          const float qv = __int_as_float(en.y);
          const uint32_t sa = st_lo + 260u * (uint32_t)en.x;
          s_lo[u] = fmaf(qv, __uint_as_float(lds_u32(sa)), s_lo[u]);
          s_hi[u] = fmaf(qv, __uint_as_float(lds_u32(sa + 128u)), s_hi[u]);
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < kVGroup; ++u) {
        if (u >= cols) break;
        for (int l = 0; l < k; ++l) {
          const int2 en = lds_i2(ebuf_a + 8u * (uint32_t)(u * k + l));
          const float qv = __int_as_float(en.y);
          const uint32_t sa = st_lo + 260u * (uint32_t)en.x;
          s_lo[u] = fmaf(qv, __uint_as_float(lds_u32(sa)), s_lo[u]);
          s_hi[u] = fmaf(qv, __uint_as_float(lds_u32(sa + 128u)), s_hi[u]);
        }
      }
    }
    if (vec && cols == kVGroup) {
      if (on_lo) {
        *reinterpret_cast<float4*>(v_lo + j0) = make_float4(s_lo[0], s_lo[1], s_lo[2], s_lo[3]);
        *reinterpret_cast<float4*>(v_lo + j0 + 4) = make_float4(s_lo[4], s_lo[5], s_lo[6], s_lo[7]);
      }
      if (on_hi) {
        *reinterpret_cast<float4*>(v_hi + j0) = make_float4(s_hi[0], s_hi[1], s_hi[2], s_hi[3]);
        *reinterpret_cast<float4*>(v_hi + j0 + 4) = make_float4(s_hi[4], s_hi[5], s_hi[6], s_hi[7]);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kVGroup; ++u) {
        if (u < cols) {
          if (on_lo) v_lo[j0 + u] = s_lo[u];
          if (on_hi) v_hi[j0 + u] = s_hi[u];
        }
      }
    }
  }
}

// dst[c][a] = src[a][c] for a d x d fp32 matrix, 32 x 32 tiles through
// padded shared memory (both sides coalesced).
__global__ void k_transpose_dd(const float* __restrict__ src, int d, float* __restrict__ dst) {
  __shared__ float t[32][33];
  griddep_launch_dependents();
  griddep_wait();                // src is dS from the compressed step
  const int c0 = blockIdx.x * 32, a0 = blockIdx.y * 32;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int a = a0 + r, c = c0 + threadIdx.x;
    t[r][threadIdx.x] = (a < d && c < d) ? src[(int64_t)a * d + c] : 0.0f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int c = c0 + r, a = a0 + threadIdx.x;
    if (c < d && a < d) dst[(int64_t)c * d + a] = t[threadIdx.x][r];
  }
}

// V[a][j] = sum_l q_{j,l} dS[a][c_{j,l}] (k = 8) reading dS^T (dst[c][a])
// straight from L1 / L2, with no staging: lanes along a (two rows a each, a
// warp covers 64 consecutive a), so every entry is one 256-byte load of a
// row segment of dS^T; a warp takes 8 columns j at a time (the entries are
// warp-uniform 32-byte loads of Q's ELL rows, all 64 row loads of a group in
// flight) and writes each a's 8 values as one 32-byte segment of V's row.
// The sums run over l in order from zero, the same as k_v.
constexpr int kVrWarps = 8, kVrGroupsPerWarp = 1;
__global__ void __launch_bounds__(32 * kVrWarps) k_v_rows(const float* __restrict__ dSt, int d,
                                                          const int32_t* __restrict__ qidx,
                                                          const float* __restrict__ qval, int64_t n,
                                                          float* __restrict__ V) {
  __shared__ int2 ebuf_all[kVrWarps][kVGroup * 8];
  griddep_launch_dependents();
  griddep_wait();                // dS^T comes from the transpose
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int2* ebuf = ebuf_all[warp];
  const uint32_t ebuf_a = smem_u32(ebuf);
  const int a = blockIdx.y * 64 + 2 * lane;         // this lane's rows a, a + 1 (d % 64 == 0)
  const int64_t n_groups = n / kVGroup;
  const float* drow = dSt + a;
  for (int64_t g = (int64_t)blockIdx.x * kVrWarps + warp; g < n_groups; g += (int64_t)gridDim.x * kVrWarps) {
    const int64_t j0 = g * kVGroup;
    // the group's 64 entries (8 columns x 8) through the warp's buffer: one
    // coalesced 8-byte load of ids and of values per lane
    const int2 ids = __ldg(reinterpret_cast<const int2*>(qidx + j0 * 8) + lane);
    const float2 vals = __ldg(reinterpret_cast<const float2*>(qval + j0 * 8) + lane);
    __syncwarp();
    ebuf[2 * lane] = make_int2(ids.x, __float_as_int(vals.x));
    ebuf[2 * lane + 1] = make_int2(ids.y, __float_as_int(vals.y));
    __syncwarp();
    float2 acc[kVGroup];
#pragma unroll
    for (int ub = 0; ub < kVGroup; ub += 2) {
      // two columns' 16 row loads in flight at once
      float2 x[2][8];
      float q[2][8];
#pragma unroll
      for (int uu = 0; uu < 2; ++uu)
#pragma unroll
        for (int l = 0; l < 8; ++l) {
          const int2 en = lds_i2(ebuf_a + 8u * (uint32_t)((ub + uu) * 8 + l));
          q[uu][l] = __int_as_float(en.y);
          x[uu][l] = __ldg(reinterpret_cast<const float2*>(drow + (int64_t)en.x * d));
        }
#pragma unroll
      for (int uu = 0; uu < 2; ++uu) {
        float2 sacc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int l = 0; l < 8; ++l) {
          sacc.x = fmaf(q[uu][l], x[uu][l].x, sacc.x);
          sacc.y = fmaf(q[uu][l], x[uu][l].y, sacc.y);
        }
        acc[ub + uu] = sacc;
      }
    }
    float* v0r = V + (int64_t)a * n + j0;
    float* v1r = v0r + n;
    *reinterpret_cast<float4*>(v0r) = make_float4(acc[0].x, acc[1].x, acc[2].x, acc[3].x);
    *reinterpret_cast<float4*>(v0r + 4) = make_float4(acc[4].x, acc[5].x, acc[6].x, acc[7].x);
    *reinterpret_cast<float4*>(v1r) = make_float4(acc[0].y, acc[1].y, acc[2].y, acc[3].y);
    *reinterpret_cast<float4*>(v1r + 4) = make_float4(acc[4].y, acc[5].y, acc[6].y, acc[7].y);
  }
}

__global__ void k_v_generic(const float* __restrict__ dS, int d, const int32_t* __restrict__ qidx,
                            const float* __restrict__ qval, int k, int64_t n, float* __restrict__ V) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)d * n) return;
  const int64_t j = t % n;
  const int a = (int)(t / n);
  float acc = 0.0f;
  for (int l = 0; l < k; ++l) acc = fmaf(qval[j * k + l], dS[(int64_t)a * d + qidx[j * k + l]], acc);
  V[(int64_t)a * n + j] = acc;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

// W[i][j] -= sum_l p_{i,l} V[a_{i,l}][j]; persistent CTAs over (column block, row) work.
// A 64-column block of V sits in shared memory (vs[a * 64 + jj]); each warp
// takes groups of R rows whose R*k <= 32 projector entries are fetched with
// one coalesced load per lane, one group ahead, staged in a per-warp buffer
// and read back as warp-uniform broadcasts.  W is read and written once,
// two columns per lane.
constexpr int kApplyMaxR = 8;

template <bool kBf16W>
__global__ void __launch_bounds__(512) k_apply(const float* __restrict__ V, int d, int64_t n, int64_t m,
                                               const int32_t* __restrict__ pidx, const float* __restrict__ pval,
                                               int k, int R, void* __restrict__ W, uint16_t* __restrict__ mirror,
                                               int64_t total_items, int64_t items_per_cta, int vec_ok) {
  extern __shared__ float vs[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  int2* ebuf = reinterpret_cast<int2*>(vs + (size_t)d * kApplyCols) + warp * 32;
  int64_t cur = (int64_t)blockIdx.x * items_per_cta;
  const int64_t end = min(total_items, cur + items_per_cta);
  const int ne = R * k;
  while (cur < end) {
    const int64_t jb = cur / m;
    const int64_t i_begin = cur % m;
    const int64_t i_end = min(m, i_begin + (end - cur));
    const int64_t j0 = jb * kApplyCols;
    __syncthreads();
    for (int e = threadIdx.x; e < d * kApplyCols; e += blockDim.x) {
      const int a = e / kApplyCols, jj = e % kApplyCols;
      vs[e] = (j0 + jj < n) ? V[(int64_t)a * n + j0 + jj] : 0.0f;
    }
    __syncthreads();
    const int64_t j = j0 + 2 * lane;
    const bool on0 = j < n, on1 = j + 1 < n;
    const bool vec = vec_ok && on1;
    int64_t ib = i_begin + (int64_t)warp * R;
    const int64_t stride = (int64_t)nwarps * R;
    // entries of the first group
    int2 pre = make_int2(0, 0);
    if (ib < i_end && lane < ne && ib + lane / k < i_end)
      pre = make_int2(pidx[ib * k + lane], __float_as_int(pval[ib * k + lane]));
    for (; ib < i_end; ib += stride) {
      __syncwarp();
      ebuf[lane] = pre;
      __syncwarp();
      const int64_t nb = ib + stride;
      if (nb < i_end && lane < ne && nb + lane / k < i_end)
        pre = make_int2(pidx[nb * k + lane], __float_as_int(pval[nb * k + lane]));
      float w0[kApplyMaxR], w1[kApplyMaxR];
#pragma unroll
      for (int r = 0; r < kApplyMaxR; ++r) {
        const int64_t i = ib + r;
        w0[r] = w1[r] = 0.0f;
        if (r >= R || i >= i_end) continue;
        const int64_t off = i * n + j;
        if (kBf16W) {
          const uint16_t* Wb = static_cast<const uint16_t*>(W);
          if (vec) {
            const uint32_t u = *reinterpret_cast<const uint32_t*>(Wb + off);
            w0[r] = __uint_as_float(u << 16);
            w1[r] = __uint_as_float(u & 0xFFFF0000u);
          } else {
            if (on0) w0[r] = __uint_as_float((uint32_t)Wb[off] << 16);
            if (on1) w1[r] = __uint_as_float((uint32_t)Wb[off + 1] << 16);
          }
        } else {
          const float* Wf = static_cast<const float*>(W);
          if (vec) {
            const float2 u = *reinterpret_cast<const float2*>(Wf + off);
            w0[r] = u.x;
            w1[r] = u.y;
          } else {
            if (on0) w0[r] = Wf[off];
            if (on1) w1[r] = Wf[off + 1];
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kApplyMaxR; ++r) {
        const int64_t i = ib + r;
        if (r >= R || i >= i_end) continue;
        float s0 = 0.0f, s1 = 0.0f;
        for (int l = 0; l < k; ++l) {
          const int2 en = ebuf[r * k + l];
          const float p = __int_as_float(en.y);
          const float2 v = *reinterpret_cast<const float2*>(vs + en.x * kApplyCols + 2 * lane);
          s0 = fmaf(p, v.x, s0);
          s1 = fmaf(p, v.y, s1);
        }
        const float n0 = w0[r] - s0, n1 = w1[r] - s1;
        const int64_t off = i * n + j;
        if (kBf16W) {
          uint16_t* Wb = static_cast<uint16_t*>(W);
          if (vec) {
            *reinterpret_cast<uint32_t*>(Wb + off) =
                (uint32_t)f32_to_bf16_bits(n0) | ((uint32_t)f32_to_bf16_bits(n1) << 16);
          } else {
            if (on0) Wb[off] = f32_to_bf16_bits(n0);
            if (on1) Wb[off + 1] = f32_to_bf16_bits(n1);
          }
        } else {
          float* Wf = static_cast<float*>(W);
          if (vec) {
            *reinterpret_cast<float2*>(Wf + off) = make_float2(n0, n1);
            if (mirror)
              *reinterpret_cast<uint32_t*>(mirror + off) =
                  (uint32_t)f32_to_bf16_bits(n0) | ((uint32_t)f32_to_bf16_bits(n1) << 16);
          } else {
            if (on0) {
              Wf[off] = n0;
              if (mirror) mirror[off] = f32_to_bf16_bits(n0);
            }
            if (on1) {
              Wf[off + 1] = n1;
              if (mirror) mirror[off + 1] = f32_to_bf16_bits(n1);
            }
          }
        }
      }
    }
    cur += i_end - i_begin;
  }
}

// TMA-streamed apply: the same arithmetic as k_apply, but W arrives in
// 64 x 64 tiles and P's rows in 64-row blocks through a ring of shared-memory
// stages fed by one producer warp (2D TMA for W, 1D bulk copies for the
// entries), so every SM keeps tens of KB of HBM reads in flight.  16
// consumer warps each take 4 rows of a tile (2 columns per lane); results
// go straight to global memory with coalesced stores.  The V block is
// restaged when a CTA's work crosses into the next column block.
constexpr int kApplyRows = 64;
constexpr int kApplyConsumerWarps = 16;
constexpr int kApplyMaxStages = 4;

struct ApplyArgs {
  const float* V;
  const int32_t* pidx;
  const float* pval;
  void* W;
  uint16_t* mirror;
  int64_t n, m;
  int64_t n_rt;          // row tiles
  int64_t total;         // column blocks x row tiles
  int64_t per_cta;
  int32_t d, k;
  int32_t tile_bytes;    // 64 x 64 x element size
  int32_t ent_stride;    // bytes reserved for one entry array of a stage
  int32_t stage_stride;
  int32_t stages;
  int32_t vs_bytes;      // bytes of the V block (1024-aligned)
  int32_t vec_ok;
  int32_t v_vec;         // V rows can be read as float4 (n % 4 == 0, 16-byte aligned V)
};

template <bool kBf16W>
__global__ void __launch_bounds__(32 * (kApplyConsumerWarps + 1), 1)
    k_apply_tma(const __grid_constant__ CUtensorMap wmap, const ApplyArgs A) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // round up to 1024 with arithmetic on the __shared__ array itself, so the
  // compiler keeps the shared address space (plain LDS, not generic loads)
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* vs = reinterpret_cast<float*>(smem);
  unsigned char* stages = smem + A.vs_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + (size_t)A.stages * A.stage_stride);
  uint64_t* empty = full + kApplyMaxStages;
  int32_t* shared_flags = reinterpret_cast<int32_t*>(empty + kApplyMaxStages);   // [0] issued, [1] failed
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = A.stages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kApplyConsumerWarps);
    }
    shared_flags[0] = 0;
    shared_flags[1] = 0;
    fence_mbar_init_cluster();
  }
  __syncthreads();
  griddep_launch_dependents();
  griddep_wait();                // V, W and P may be written by earlier kernels in the stream
  const int64_t it0 = (int64_t)blockIdx.x * A.per_cta;
  const int64_t nit = imax64(0, imin64(A.total, it0 + A.per_cta) - it0);
  const int k = A.k;

  if (warp == kApplyConsumerWarps) {
    // producer
    if (lane == 0) {
      int64_t q = 0;
      int s = 0;                 // stage and ring-pass parity, advanced without divisions
      uint32_t pass = 0;
      int64_t jb = it0 / A.n_rt, rt = it0 % A.n_rt;
      for (; q < nit; ++q) {
        if (q >= S && !mbar_wait(&empty[s], pass ^ 1u)) {
          shared_flags[1] = 1;
          break;
        }
        const int rows_here = (int)imin64(kApplyRows, A.m - rt * kApplyRows);
        const uint32_t eb = (uint32_t)((rows_here * k * 4 + 15) / 16 * 16);
        unsigned char* st = stages + (size_t)s * A.stage_stride;
        mbar_arrive_expect_tx(&full[s], (uint32_t)A.tile_bytes + 2 * eb);
        tma_load_2d(st, &wmap, &full[s], (int)(jb * kApplyCols), (int)(rt * kApplyRows));
        bulk_load(st + A.tile_bytes, A.pidx + rt * kApplyRows * k, eb, &full[s]);
        bulk_load(st + A.tile_bytes + A.ent_stride, A.pval + rt * kApplyRows * k, eb, &full[s]);
        if (++s == S) {
          s = 0;
          pass ^= 1u;
        }
        if (++rt == A.n_rt) {
          rt = 0;
          ++jb;
        }
      }
      shared_flags[0] = (int32_t)q;
    }
  } else {
    // consumers
    int64_t cur_jb = -1;
    bool failed = false;
    const uint32_t stages_base = smem_u32(stages);
    const uint32_t vs_lane = smem_u32(vs) + 8u * (uint32_t)lane;
    int s = 0;
    uint32_t pass = 0;
    int64_t jb = it0 / A.n_rt, rt = it0 % A.n_rt;
    for (int64_t q = 0; q < nit; ++q) {
      if (q > 0 && ++rt == A.n_rt) {
        rt = 0;
        ++jb;
      }
      const int64_t j0 = jb * kApplyCols;
      if (jb != cur_jb) {
        named_bar_sync(1, 32 * kApplyConsumerWarps);
        if (A.v_vec && j0 + kApplyCols <= A.n) {
          // 16-byte loads, 8 in flight per thread before their stores
          constexpr int kQuads = kApplyCols / 4;               // float4 per V row of the block
          const int total4 = A.d * kQuads;
          for (int e0 = threadIdx.x; e0 < total4; e0 += 8 * 32 * kApplyConsumerWarps) {
            float4 t[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int e = e0 + u * 32 * kApplyConsumerWarps;
              if (e < total4)
                t[u] = *reinterpret_cast<const float4*>(A.V + (int64_t)(e / kQuads) * A.n + j0 + 4 * (e % kQuads));
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int e = e0 + u * 32 * kApplyConsumerWarps;
              if (e < total4) reinterpret_cast<float4*>(vs)[e] = t[u];
            }
          }
        } else {
          for (int e = threadIdx.x; e < A.d * kApplyCols; e += 32 * kApplyConsumerWarps) {
            const int a = e / kApplyCols, jj = e % kApplyCols;
            vs[e] = (j0 + jj < A.n) ? A.V[(int64_t)a * A.n + j0 + jj] : 0.0f;
          }
        }
        named_bar_sync(1, 32 * kApplyConsumerWarps);
        cur_jb = jb;
      }
      const int cur_s = s;
      const uint32_t cur_pass = pass;
      if (++s == S) {
        s = 0;
        pass ^= 1u;
      }
      if (!failed && !mbar_wait(&full[cur_s], cur_pass)) {
        failed = true;
        shared_flags[1] = 1;
      }
      if (failed) continue;
      // 32-bit shared addresses: W tile row r at st + r * 64 * esize, entry
      // arrays after it, V block row a at vs_lane + a * 256
      const uint32_t st = stages_base + (uint32_t)cur_s * (uint32_t)A.stage_stride;
      const uint32_t eidx = st + (uint32_t)A.tile_bytes;
      const uint32_t evals = eidx + (uint32_t)A.ent_stride;
      const int64_t j = j0 + 2 * lane;
      const bool on0 = j < A.n, on1 = j + 1 < A.n;
      const bool vec = A.vec_ok && on1;
      // W row r of this tile as two fp32 values
      auto w_load = [&](int r, float& w0, float& w1) {
        if (kBf16W) {
          const uint32_t u = lds_u32(st + ((uint32_t)r * kApplyCols + 2u * lane) * 2u);
          w0 = __uint_as_float(u << 16);
          w1 = __uint_as_float(u & 0xFFFF0000u);
        } else {
          const float2 u = lds_f2(st + ((uint32_t)r * kApplyCols + 2u * lane) * 4u);
          w0 = u.x;
          w1 = u.y;
        }
      };
      auto w_store = [&](int64_t i, float n0, float n1) {
        const int64_t off = i * A.n + j;
        if (kBf16W) {
          uint16_t* Wb = static_cast<uint16_t*>(A.W);
          if (vec) {
            __nv_bfloat162 h = __floats2bfloat162_rn(n0, n1);
            *reinterpret_cast<uint32_t*>(Wb + off) = *reinterpret_cast<uint32_t*>(&h);
          } else {
            if (on0) Wb[off] = f32_to_bf16_bits(n0);
            if (on1) Wb[off + 1] = f32_to_bf16_bits(n1);
          }
        } else {
          float* Wf = static_cast<float*>(A.W);
          if (vec) {
            *reinterpret_cast<float2*>(Wf + off) = make_float2(n0, n1);
            if (A.mirror) {
              __nv_bfloat162 h = __floats2bfloat162_rn(n0, n1);
              *reinterpret_cast<uint32_t*>(A.mirror + off) = *reinterpret_cast<uint32_t*>(&h);
            }
          } else {
            if (on0) {
              Wf[off] = n0;
              if (A.mirror) A.mirror[off] = f32_to_bf16_bits(n0);
            }
            if (on1) {
              Wf[off + 1] = n1;
              if (A.mirror) A.mirror[off + 1] = f32_to_bf16_bits(n1);
            }
          }
        }
      };
      const int64_t i_first = rt * kApplyRows + warp * 4;
      if (kBf16W && k == 8 && i_first + 3 < A.m && A.vec_ok && j0 + kApplyCols <= A.n) {
        // bf16 W, whole tile row in range: two rows at a time, every load
        // issued before the multiply-adds, both columns of a lane as one
        // packed pair (fused multiply-add, subtraction and rounding to bf16
        // on the pair), one 4-byte store per lane and row
        uint32_t* wrow = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(A.W) + i_first * A.n + j);
        const int64_t wstride = A.n / 2;   // 32-bit words per W row
#pragma unroll
        for (int rp = 0; rp < 4; rp += 2) {
          const int r0 = warp * 4 + rp;
          const uint32_t e0 = eidx + (uint32_t)r0 * 32u, v0a = evals + (uint32_t)r0 * 32u;
          const int4 a0 = lds_i4(e0), a1 = lds_i4(e0 + 16), a2 = lds_i4(e0 + 32), a3 = lds_i4(e0 + 48);
          const float4 p0 = lds_f4(v0a), p1 = lds_f4(v0a + 16), p2 = lds_f4(v0a + 32), p3 = lds_f4(v0a + 48);
          const uint32_t ua = lds_u32(st + ((uint32_t)r0 * kApplyCols + 2u * lane) * 2u);
          const uint32_t ub = lds_u32(st + ((uint32_t)(r0 + 1) * kApplyCols + 2u * lane) * 2u);
          const int ia[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          const int ib[8] = {a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
          const float pa[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
          const float pb[8] = {p2.x, p2.y, p2.z, p2.w, p3.x, p3.y, p3.z, p3.w};
          uint64_t va[8], vb[8];
#pragma unroll
          for (int l = 0; l < 8; ++l) {
            va[l] = lds_u64(vs_lane + (uint32_t)ia[l] * (kApplyCols * 4u));
            vb[l] = lds_u64(vs_lane + (uint32_t)ib[l] * (kApplyCols * 4u));
          }
          uint64_t sa = 0ull, sb = 0ull;
#pragma unroll
          for (int l = 0; l < 8; ++l) {
            ffma2(sa, va[l], pack_f2(pa[l], pa[l]));
            ffma2(sb, vb[l], pack_f2(pb[l], pb[l]));
          }
          const uint64_t wa = pack_f2(__uint_as_float(ua << 16), __uint_as_float(ua & 0xFFFF0000u));
          const uint64_t wb = pack_f2(__uint_as_float(ub << 16), __uint_as_float(ub & 0xFFFF0000u));
          wrow[rp * wstride] = bf16x2_rn(fsub2(wa, sa));
          wrow[(rp + 1) * wstride] = bf16x2_rn(fsub2(wb, sb));
        }
      } else if (k == 8 && i_first + 3 < A.m) {
        // two rows at a time, every load issued before the multiply-adds
#pragma unroll
        for (int rp = 0; rp < 4; rp += 2) {
          const int r0 = warp * 4 + rp;
          const uint32_t e0 = eidx + (uint32_t)r0 * 32u, v0a = evals + (uint32_t)r0 * 32u;
          const int4 a0 = lds_i4(e0), a1 = lds_i4(e0 + 16), a2 = lds_i4(e0 + 32), a3 = lds_i4(e0 + 48);
          const float4 p0 = lds_f4(v0a), p1 = lds_f4(v0a + 16), p2 = lds_f4(v0a + 32), p3 = lds_f4(v0a + 48);
          float wa0, wa1, wb0, wb1;
          w_load(r0, wa0, wa1);
          w_load(r0 + 1, wb0, wb1);
          const int ia[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          const int ib[8] = {a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
          const float pa[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
          const float pb[8] = {p2.x, p2.y, p2.z, p2.w, p3.x, p3.y, p3.z, p3.w};
          float2 va[8], vb[8];
#pragma unroll
          for (int l = 0; l < 8; ++l) {
            va[l] = lds_f2(vs_lane + (uint32_t)ia[l] * (kApplyCols * 4u));
            vb[l] = lds_f2(vs_lane + (uint32_t)ib[l] * (kApplyCols * 4u));
          }
          float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
          for (int l = 0; l < 8; ++l) {
            sa0 = fmaf(pa[l], va[l].x, sa0);
            sa1 = fmaf(pa[l], va[l].y, sa1);
            sb0 = fmaf(pb[l], vb[l].x, sb0);
            sb1 = fmaf(pb[l], vb[l].y, sb1);
          }
          w_store(i_first + rp, wa0 - sa0, wa1 - sa1);
          w_store(i_first + rp + 1, wb0 - sb0, wb1 - sb1);
        }
      } else {
        for (int r4 = 0; r4 < 4; ++r4) {
          const int r = warp * 4 + r4;
          const int64_t i = rt * kApplyRows + r;
          if (i >= A.m) break;
          float w0, w1;
          w_load(r, w0, w1);
          float s0 = 0.0f, s1 = 0.0f;
          const uint32_t ri = eidx + (uint32_t)(r * k) * 4u;
          const uint32_t rv = evals + (uint32_t)(r * k) * 4u;
          for (int l = 0; l < k; ++l) {
            const int a = (int)lds_u32(ri + 4u * l);
            const float p = __uint_as_float(lds_u32(rv + 4u * l));
            const float2 v = lds_f2(vs_lane + (uint32_t)a * (kApplyCols * 4u));
            s0 = fmaf(p, v.x, s0);
            s1 = fmaf(p, v.y, s1);
          }
          w_store(i, w0 - s0, w1 - s1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_local(&empty[cur_s]);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && shared_flags[1]) {
    // a wait ran out: let the copies still in flight land (bounded) before exit
    const int64_t issued = shared_flags[0];
    for (int64_t q = imax64(0, issued - S); q < issued; ++q)
      mbar_wait(&full[q % S], (uint32_t)(q / S) & 1u);
  }
}

template <bool kBf16W>
__global__ void k_apply_generic(const float* __restrict__ V, int64_t n, int64_t m, const int32_t* __restrict__ pidx,
                                const float* __restrict__ pval, int k, void* __restrict__ W,
                                uint16_t* __restrict__ mirror) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= m * n) return;
  const int64_t i = t / n, j = t % n;
  float s = 0.0f;
  for (int l = 0; l < k; ++l) s = fmaf(pval[i * k + l], V[(int64_t)pidx[i * k + l] * n + j], s);
  if (kBf16W) {
    uint16_t* Wb = static_cast<uint16_t*>(W);
    Wb[t] = f32_to_bf16_bits(__uint_as_float((uint32_t)Wb[t] << 16) - s);
  } else {
    float* Wf = static_cast<float*>(W);
    const float nv = Wf[t] - s;
    Wf[t] = nv;
    if (mirror) mirror[t] = f32_to_bf16_bits(nv);
  }
}

}  // namespace

// ----------------------------------------------------------------------------
// Host side (declared in lsp_internal.cuh)
// ----------------------------------------------------------------------------

GatherPlan plan_gather(int64_t rows, int64_t ncols, int d) {
  GatherPlan p;
  // the projector's output range (a_rng = 8 x min(16, ceil(d / 8))), kGatherOut per warp
  p.warps = 8 * std::min(16, (d + 7) / 8) / kGatherOut;
  p.n_ar = (d + kGatherOut * p.warps - 1) / (kGatherOut * p.warps);
  p.n_cb = (int)ceil_div<int64_t>(ncols, kColsPerCta);
  p.n_win = (int)ceil_div<int64_t>(rows, kWinRows);
  const int64_t base = (int64_t)p.n_cb * p.n_ar;
  int splits = (int)std::max<int64_t>(1, std::min<int64_t>(p.n_win, kTargetCtas / std::max<int64_t>(1, base)));
  p.win_per_split = (int)ceil_div<int64_t>(p.n_win, splits);
  p.splits = (int)ceil_div<int64_t>(p.n_win, p.win_per_split);
  p.partial_bytes = p.splits > 1 ? align_up((size_t)p.splits * ncols * d * 4, 256) : 0;
  // more tiles than one wave: whole waves of whole tiles, then the column
  // blocks left over split by windows when that at least halves the last
  // wave's length (a pure function of the sizes, like the rest)
  p.cb_main = p.n_cb;
  p.tail_splits = 1;
  p.tail_wps = p.n_win;
  if (p.splits == 1 && base > kWaveCtas && kWaveCtas % p.n_ar == 0) {
    const int64_t cb_main = base / kWaveCtas * (kWaveCtas / p.n_ar);
    const int64_t tail_tiles = (p.n_cb - cb_main) * p.n_ar;
    const int64_t ts = tail_tiles > 0 ? std::min<int64_t>(p.n_win, kWaveCtas / tail_tiles) : 1;
    if (ts >= 2) {
      p.cb_main = (int)cb_main;
      p.tail_wps = (int)ceil_div<int64_t>(p.n_win, ts);
      p.tail_splits = (int)ceil_div<int64_t>(p.n_win, p.tail_wps);
      const int64_t tail_cols = ncols - cb_main * kColsPerCta;
      p.partial_bytes = align_up((size_t)(p.tail_splits - 1) * tail_cols * d * 4, 256);
    }
  }
  return p;
}


CompressPlan plan_compress(int64_t m, int64_t n, int d) {
  CompressPlan c;
  c.g1 = plan_gather(m, n, d);
  c.g2 = plan_gather(n, d, d);
  // stage 2 reads R^T (at the workspace's 256-byte aligned start) with the
  // row gather whenever its rows are 16-byte multiples; only otherwise does
  // it take the staged gather, whose row splits need partials
  c.stage2_rows = d % 4 == 0;
  size_t off = 0;
  c.off_rt = off;
  off = align_up(off + (size_t)n * d * 4, 256);
  c.off_rtp = off;
  off += c.g1.partial_bytes;
  c.off_sp = off;
  if (!c.stage2_rows) off += c.g2.partial_bytes;
  c.bytes = off;
  return c;
}

// V (d x n fp32), then dS^T (d x d fp32) for the row-gather form of V.
size_t decompress_bytes(int64_t n, int d) { return align_up((size_t)d * n * 4, 256) + align_up((size_t)d * d * 4, 256); }

constexpr size_t kMaxGatherSmem = 220 * 1024;

size_t gather_stage_bytes(const lsp_projector_s* Ap, size_t es) {
  const size_t tile = (size_t)kWinRows * kColsPerCta * es;
  return align_up(align_up(align_up(tile, 128) + 16 * 40, 128) + (size_t)Ap->max_slice_bytes, 1024);
}

size_t gather_smem_estimate(const lsp_projector_s* Ap, size_t es) {
  return 2 * gather_stage_bytes(Ap, es) + 2048;   // the ring needs at least two stages
}

// A tensor map may be built on B: 16-byte aligned base and rows, and B in
// the current device's memory (anything else takes the plain-load kernels).
bool tma_ok(const void* B, int64_t ldb, size_t esize) {
  return (reinterpret_cast<uintptr_t>(B) % 16) == 0 && (ldb * (int64_t)esize) % 16 == 0 &&
         tensor_map_encoder() != nullptr && on_current_device(B);
}

// The staged gather's launch for one matrix: its arguments, tensor map,
// dynamic shared memory and block count.  Returns false when the shape or
// the operand's placement needs the plain-load kernel instead.
struct GatherLaunch {
  GatherArgs A;
  CUtensorMap map;
  size_t smem;
  int blocks;           // on a 1D grid
  dim3 grid;            // the same blocks as this launch's own grid
  int block_threads;
  bool tail;
};

template <typename TB>
sf_status prepare_gather(const lsp_projector_s* Aproj, const TB* B, int64_t ldb, int64_t ncols, const GatherPlan& p,
                         float* yt_final, float* yt_partial, GatherLaunch* L, bool* staged) {
  const int64_t rows = Aproj->rows;
  const int d = Aproj->d;
  const size_t es = sizeof(TB);
  *staged = tma_ok(B, ldb, es) && Aproj->a_rng == kGatherOut * p.warps &&
            gather_smem_estimate(Aproj, es) <= kMaxGatherSmem;
  if (!*staged) return SF_OK;
  const int align_elems = (int)(16 / es);
  const int cbx = (int)std::min<int64_t>(kColsPerCta, ceil_div<int64_t>(ncols, align_elems) * align_elems);
  GatherArgs& A = L->A;
  A.wptr = Aproj->wptr;
  A.went = Aproj->went;
  A.gdesc = Aproj->gdesc;
  const bool tail = p.tail_splits > 1;
  const int64_t tail_c0 = (int64_t)p.cb_main * kColsPerCta;
  A.yt = yt_final;
  A.part = yt_partial;
  A.direct0 = p.splits > 1 ? 0 : 1;
  A.split_stride = tail ? (ncols - tail_c0) * d : ncols * d;
  A.out_c0 = tail ? (int32_t)tail_c0 : 0;
  A.main_tiles = tail ? p.cb_main * p.n_ar : 0;
  A.cb_main = p.cb_main;
  A.n_cb = p.n_cb;
  A.n_ar = p.n_ar;
  A.tail_wps = p.tail_wps;
  A.ncols = (int32_t)ncols;
  A.d = d;
  A.dp = Aproj->dp;
  A.n_win = p.n_win;
  A.win_per_split = p.win_per_split;
  A.cbx = cbx;
  A.stage_tx = kWinRows * cbx * (int)es;
  A.wsl_off = (int)align_up((size_t)A.stage_tx, 128);
  A.wbytes = (int)align_up((size_t)(kGatherOut * p.warps + 1) * 4, 16);
  A.ent_off = (int)align_up((size_t)A.wsl_off + A.wbytes, 128);
  A.stage_stride = (int)align_up((size_t)A.ent_off + Aproj->max_slice_bytes, 1024);
  A.stages = (int)std::min<size_t>(kMaxStages, (kMaxGatherSmem - 2048) / A.stage_stride);
  A.vec_out = (d % 4 == 0) && (reinterpret_cast<uintptr_t>(A.yt) % 16 == 0) ? 1 : 0;

  cuuint64_t dims[2] = {(cuuint64_t)ncols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ldb * (int64_t)es)};
  cuuint32_t box[2] = {(cuuint32_t)cbx, (cuuint32_t)kWinRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = tensor_map_encoder()(&L->map, es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                    2, const_cast<TB*>(B), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SF_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  L->smem = (size_t)A.stages * A.stage_stride + 2 * kMaxStages * sizeof(uint64_t) + kMaxStages * 4 + 8 + 1024;
  L->tail = tail;
  L->blocks = tail ? A.main_tiles + (p.n_cb - p.cb_main) * p.n_ar * p.tail_splits : p.n_cb * p.n_ar * p.splits;
  L->grid = tail ? dim3((unsigned)L->blocks) : dim3((unsigned)p.n_cb, (unsigned)p.n_ar, (unsigned)p.splits);
  L->block_threads = 32 * p.warps;
  return SF_OK;
}

// After the gather kernel: the split tail's partials added into Y^T, or the
// row splits' partials reduced into it.
sf_status finish_gather(const GatherPlan& p, int64_t ncols, int d, float* yt_final, float* yt_partial,
                        cudaStream_t stream) {
  if (p.tail_splits > 1) {
    const int64_t tail_c0 = (int64_t)p.cb_main * kColsPerCta;
    const int64_t n_out = (ncols - tail_c0) * d;
    const int blocks = (int)std::min<int64_t>(ceil_div<int64_t>(n_out, 256), (int64_t)sm_count() * 4);
    SF_CUDA_TRY(launch_pdl(k_add_splits, dim3(blocks), dim3(256), 0, stream, yt_partial, p.tail_splits - 1,
                           n_out, n_out, yt_final + tail_c0 * d),
                "launch k_add_splits");
  } else if (p.splits > 1) {
    const int64_t n_out = ncols * d;
    const int blocks = (int)std::min<int64_t>(ceil_div<int64_t>(n_out, 256), (int64_t)sm_count() * 4);
    SF_CUDA_TRY(launch_pdl(k_reduce_splits, dim3(blocks), dim3(256), 0, stream, yt_partial, p.splits, n_out, n_out,
                           yt_final),
                "launch k_reduce_splits");
  }
  return SF_OK;
}

template <typename TB>
sf_status launch_generic_gather(const lsp_projector_s* Aproj, const TB* B, int64_t ldb, int64_t ncols, float* yt_final,
                                cudaStream_t stream) {
  const int64_t total = ncols * Aproj->d;
  k_gather_generic<TB><<<(unsigned)ceil_div<int64_t>(total, 256), 256, 0, stream>>>(
      B, ldb, ncols, Aproj->d, Aproj->col_ptr, Aproj->row_idx, Aproj->csc_val, yt_final);
  return check_launch("k_gather_generic");
}

cudaLaunchConfig_t pdl_config(dim3 grid, int threads, size_t smem, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <typename TB>
sf_status launch_gather(const lsp_projector_s* Aproj, const TB* B, int64_t ldb, int64_t ncols, const GatherPlan& p,
                        float* yt_final, float* yt_partial, cudaStream_t stream) {
  GatherLaunch L;
  bool staged = false;
  SF_TRY(prepare_gather<TB>(Aproj, B, ldb, ncols, p, yt_final, yt_partial, &L, &staged));
  if (!staged) return launch_generic_gather<TB>(Aproj, B, ldb, ncols, yt_final, stream);
  SF_TRY(allow_dynamic_smem(reinterpret_cast<const void*>(&k_gather_t<TB>), kMaxGatherSmem));
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(L.grid, L.block_threads, L.smem, stream, attr);
  SF_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_gather_t<TB>, L.map, L.A), "launch k_gather_t");
  return finish_gather(p, ncols, Aproj->d, yt_final, yt_partial, stream);
}

// The stage-1 gathers of several matrices of one element type and one block
// shape in one launch, matrices with the longest tiles first (they set the
// launch's length); each matrix's tiles, partials and sums exactly as in its
// own launch.
template <typename TB>
sf_status launch_gather_multi(int count, const lsp_projector_s* const* Aproj, const TB* const* B, const int64_t* ldb,
                              const int64_t* ncols, const GatherPlan* p, float* const* yt_final,
                              float* const* yt_partial, cudaStream_t stream) {
  std::vector<int> staged_ids;
  std::vector<GatherLaunch> L(count);
  for (int i = 0; i < count; ++i) {
    bool staged = false;
    SF_TRY(prepare_gather<TB>(Aproj[i], B[i], ldb[i], ncols[i], p[i], yt_final[i], yt_partial[i], &L[i], &staged));
    if (staged) staged_ids.push_back(i);
    else SF_TRY(launch_generic_gather<TB>(Aproj[i], B[i], ldb[i], ncols[i], yt_final[i], stream));
  }
  // longest tiles first; gathers whose block shape differs go alone
  std::stable_sort(staged_ids.begin(), staged_ids.end(), [&](int a, int b) { return p[a].n_win > p[b].n_win; });
  size_t at = 0;
  while (at < staged_ids.size()) {
    MultiGatherArgs M;
    M.count = 0;
    size_t smem = 0;
    int blocks = 0;
    const int threads = L[staged_ids[at]].block_threads;
    while (at < staged_ids.size() && M.count < kMaxLayerMats && L[staged_ids[at]].block_threads == threads) {
      const GatherLaunch& g = L[staged_ids[at]];
      M.map[M.count] = g.map;
      M.a[M.count] = g.A;
      blocks += g.blocks;
      M.block_end[M.count] = blocks;
      smem = std::max(smem, g.smem);
      ++M.count;
      ++at;
    }
    SF_TRY(allow_dynamic_smem(reinterpret_cast<const void*>(&k_gather_t_multi<TB>), kMaxGatherSmem));
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)blocks), threads, smem, stream, attr);
    SF_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_gather_t_multi<TB>, M), "launch k_gather_t_multi");
  }
  for (int i : staged_ids) SF_TRY(finish_gather(p[i], ncols[i], Aproj[i]->d, yt_final[i], yt_partial[i], stream));
  return SF_OK;
}

// Y^T = (A^T B)^T for a small L2-resident B (the second compress stage):
// k_rowgather when B's rows are 16-byte aligned, else the staged gather.
sf_status launch_stage2(const lsp_projector_s* Aproj, const float* B, int64_t ldb, int64_t ncols, const GatherPlan& p,
                        float* yt_final, float* yt_partial, cudaStream_t stream) {
  if ((reinterpret_cast<uintptr_t>(B) % 16) != 0 || ldb % 4 != 0 || ncols % 4 != 0 || ncols > INT32_MAX)
    return launch_gather<float>(Aproj, B, ldb, ncols, p, yt_final, yt_partial, stream);
  const dim3 grid((unsigned)ceil_div(Aproj->d, kRgWarps), (unsigned)ceil_div<int64_t>(ncols, kRgCols));
  SF_CUDA_TRY(launch_pdl(k_rowgather, grid, dim3(32 * kRgWarps), 0, stream, B, ldb, (int)ncols, Aproj->col_ptr,
                         Aproj->row_idx, Aproj->csc_val, Aproj->d, yt_final),
              "launch k_rowgather");
  return SF_OK;
}

// The second stage of several matrices: one k_rowgather_multi launch per
// kMaxLayerMats matrices whose Rᵀ rows are 16-byte aligned, the staged
// gather for the others.
sf_status launch_stage2_multi(int count, const lsp_projector_s* const* Aproj, const float* const* B, const int64_t* ldb,
                              const int64_t* ncols, const GatherPlan* p, float* const* yt_final,
                              float* const* yt_partial, cudaStream_t stream) {
  MultiRowGatherArgs M;
  M.count = 0;
  int blocks = 0;
  auto flush = [&]() -> sf_status {
    if (M.count == 0) return SF_OK;
    SF_CUDA_TRY(launch_pdl(k_rowgather_multi, dim3((unsigned)blocks), dim3(32 * kRgWarps), 0, stream, M),
                "launch k_rowgather_multi");
    M.count = 0;
    blocks = 0;
    return SF_OK;
  };
  for (int i = 0; i < count; ++i) {
    if ((reinterpret_cast<uintptr_t>(B[i]) % 16) != 0 || ldb[i] % 4 != 0 || ncols[i] % 4 != 0 ||
        ncols[i] > INT32_MAX) {
      SF_TRY(launch_gather<float>(Aproj[i], B[i], ldb[i], ncols[i], p[i], yt_final[i], yt_partial[i], stream));
      continue;
    }
    const int gx = ceil_div(Aproj[i]->d, kRgWarps), gy = (int)ceil_div<int64_t>(ncols[i], kRgCols);
    M.a[M.count] = RowGatherArgs{B[i], ldb[i], (int)ncols[i], Aproj[i]->col_ptr, Aproj[i]->row_idx,
                                 Aproj[i]->csc_val, Aproj[i]->d, yt_final[i]};
    M.gx[M.count] = gx;
    blocks += gx * gy;
    M.block_end[M.count] = blocks;
    if (++M.count == kMaxLayerMats) SF_TRY(flush());
  }
  return flush();
}

sf_status check_proj(const lsp_projector_s* p, const char* name) {
  if (!p) return fail(SF_ERR_INVALID, "projector %s is NULL", name);
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != p->device) return fail(SF_ERR_INVALID, "projector %s was built on device %d, current is %d", name,
                                    p->device, dev);
  return SF_OK;
}

template sf_status launch_gather<float>(const lsp_projector_s*, const float*, int64_t, int64_t, const GatherPlan&,
                                        float*, float*, cudaStream_t);
template sf_status launch_gather<__nv_bfloat16>(const lsp_projector_s*, const __nv_bfloat16*, int64_t, int64_t,
                                                const GatherPlan&, float*, float*, cudaStream_t);

// Host read-back of the device error word (used by sf_sync_status).
int read_and_clear_device_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_device_error, &z, sizeof z);
  return v;
}

}  // namespace sf

using sf::ceil_div;
using sf::fail;

extern "C" {

sf_status lsp_projector_create(int64_t rows, int32_t d, int32_t k, const int32_t* d_col_idx, const float* d_val,
                               int validate, void* stream_, lsp_projector* out) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("lsp_projector_create");
  if (!out) return fail(SF_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (rows < 1 || d < 1 || d > 1024 || k < 1 || k > 64)
    return fail(SF_ERR_INVALID, "need rows >= 1, 1 <= d <= 1024, 1 <= k <= 64 (got %lld, %d, %d)", (long long)rows,
                d, k);
  if (rows * (int64_t)k >= (int64_t)INT32_MAX) return fail(SF_ERR_UNSUPPORTED, "rows * k must be < 2^31");
  if (!d_col_idx || !d_val) return fail(SF_ERR_INVALID, "ELL arrays are NULL");
  cudaStream_t stream = sf::as_stream(stream_);
  lsp_projector_s* p = new (std::nothrow) lsp_projector_s;
  if (!p) return fail(SF_ERR_OOM, "projector allocation failed");
  cudaGetDevice(&p->device);
  p->rows = rows;
  p->d = d;
  p->k = k;
  p->dp = (d + 7) / 8 * 8;
  p->n_win = (int32_t)ceil_div<int64_t>(rows, sf::kWinRows);
  const int64_t nnz = rows * k;
  const int64_t nwd = (int64_t)p->n_win * p->dp;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = sf::align_up(off + bytes, 256);
    return o;
  };
  p->a_rng = 8 * std::min(16, (d + 7) / 8);
  p->n_ar = (int32_t)ceil_div(d, p->a_rng);
  // wptr and went are padded so the 16-byte rounded bulk copies of the
  // gather kernel never read past the allocation
  const size_t o_eidx = take(nnz * 4 + 64), o_eval = take(nnz * 4 + 64), o_cptr = take((d + 1) * 4), o_ridx = take(nnz * 4),
               o_cval = take(nnz * 4), o_perm = take(d * 4), o_wptr = take((nwd + 1 + 16) * 4),
               o_went = take((nnz + 4) * 8), o_gd = take((size_t)p->n_ar * p->n_win * 8), o_wcnt = take(nwd * 4),
               o_coff = take(nwd * 4), o_tot = take(d * 4), o_err = take(8), o_e2c = take(nnz * 4),
               o_e2w = take(nnz * 4);
  if (cudaMalloc(&p->block, off) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return fail(SF_ERR_OOM, "cudaMalloc of %zu bytes for the projector failed", off);
  }
  char* b = static_cast<char*>(p->block);
  p->ell_idx = reinterpret_cast<int32_t*>(b + o_eidx);
  p->ell_val = reinterpret_cast<float*>(b + o_eval);
  p->col_ptr = reinterpret_cast<int32_t*>(b + o_cptr);
  p->row_idx = reinterpret_cast<int32_t*>(b + o_ridx);
  p->csc_val = reinterpret_cast<float*>(b + o_cval);
  p->bucket_perm = reinterpret_cast<int32_t*>(b + o_perm);
  p->wptr = reinterpret_cast<int32_t*>(b + o_wptr);
  p->went = reinterpret_cast<int2*>(b + o_went);
  p->gdesc = reinterpret_cast<int2*>(b + o_gd);
  p->wcnt = reinterpret_cast<int32_t*>(b + o_wcnt);
  p->csc_off = reinterpret_cast<int32_t*>(b + o_coff);
  p->totals = reinterpret_cast<int32_t*>(b + o_tot);
  p->err = reinterpret_cast<int32_t*>(b + o_err);
  p->ell2csc = reinterpret_cast<int32_t*>(b + o_e2c);
  p->ell2went = reinterpret_cast<int32_t*>(b + o_e2w);

  auto bail = [&](sf_status st) {
    cudaFree(p->block);
    delete p;
    return st;
  };
  if (cudaMemsetAsync(p->err, 0, 8, stream) != cudaSuccess || cudaMemsetAsync(p->wptr + nwd + 1, 0, 64, stream) != cudaSuccess ||
      cudaMemsetAsync(p->went + nnz, 0, 32, stream) != cudaSuccess ||
      cudaMemsetAsync(p->ell2csc, 0xFF, nnz * 4, stream) != cudaSuccess ||
      cudaMemsetAsync(p->ell2went, 0xFF, nnz * 4, stream) != cudaSuccess)
    return bail(sf::cuda_fail(cudaGetLastError(), "memset"));
  const int nsm = sf::sm_count();
  sf::k_copy_ell<<<(unsigned)std::min<int64_t>(ceil_div<int64_t>(nnz, 256), nsm * 8), 256, 0, stream>>>(
      d_col_idx, d_val, nnz, d, p->ell_idx, p->ell_val);
  if (validate)
    sf::k_validate_rows<<<(unsigned)ceil_div<int64_t>(rows, 256), 256, 0, stream>>>(d_col_idx, rows, k, d, p->err);
  sf::k_window_hist<<<p->n_win, 256, p->dp * 4, stream>>>(d_col_idx, rows, k, d, p->dp, p->wcnt, p->err);
  sf::k_column_offsets<<<(unsigned)ceil_div(d, 128), 128, 0, stream>>>(p->wcnt, p->n_win, d, p->dp, p->csc_off,
                                                                      p->totals);
  sf::k_scan_exclusive<<<1, 1024, 0, stream>>>(p->totals, d, p->col_ptr);
  sf::k_scan_exclusive<<<1, 1024, 0, stream>>>(p->wcnt, nwd, p->wptr);
  const int wpb = 4;
  sf::k_place<<<(unsigned)ceil_div(p->n_win, wpb), 32 * wpb, wpb * p->dp * 4, stream>>>(
      d_col_idx, d_val, rows, k, d, p->dp, p->n_win, p->wptr, p->csc_off, p->col_ptr, p->went, p->row_idx,
      p->csc_val, p->ell2csc, p->ell2went);
  sf::k_bucket_perm<<<1, 1024, 0, stream>>>(p->col_ptr, d, p->bucket_perm);
  sf::k_gdesc<<<(unsigned)ceil_div<int64_t>((int64_t)p->n_ar * p->n_win, 256), 256, 0, stream>>>(
      p->wptr, p->n_win, p->dp, p->a_rng, p->n_ar, p->gdesc, p->err + 1);
  sf_status st = sf::check_launch("projector build");
  if (st != SF_OK) return bail(st);
  // the build ends with one bounded wait: the gather launches need the
  // largest slice size on the host
  st = sf::bounded_wait_stream(stream, 0, "lsp_projector_create");
  if (st != SF_OK) return bail(st);
  int32_t flags[2] = {0, 0};
  if (cudaMemcpy(flags, p->err, 8, cudaMemcpyDeviceToHost) != cudaSuccess)
    return bail(sf::cuda_fail(cudaGetLastError(), "read build flags"));
  p->max_slice_bytes = flags[1];
  p->bad_ids = (flags[0] & sf::kDevErrIndex) != 0;
  if (validate) {
    if (flags[0] & sf::kDevErrIndex) return bail(fail(SF_ERR_INVALID, "projector has a column id outside [0, %d)", d));
    if (flags[0] & 4) return bail(fail(SF_ERR_INVALID, "projector repeats a column id inside a row"));
  }
  *out = p;
  return SF_OK;
}

sf_status lsp_projector_export_csc(lsp_projector p, int32_t* col_ptr, int32_t* row_idx, float* val,
                                   int32_t* bucket_perm, void* stream_) {
  sf::clear_error();
  SF_TRY(sf::check_proj(p, "P"));
  cudaStream_t s = sf::as_stream(stream_);
  const size_t nnz = (size_t)p->rows * p->k;
  if (col_ptr) SF_CUDA_TRY(cudaMemcpyAsync(col_ptr, p->col_ptr, (p->d + 1) * 4, cudaMemcpyDeviceToDevice, s), "export");
  if (row_idx) SF_CUDA_TRY(cudaMemcpyAsync(row_idx, p->row_idx, nnz * 4, cudaMemcpyDeviceToDevice, s), "export");
  if (val) SF_CUDA_TRY(cudaMemcpyAsync(val, p->csc_val, nnz * 4, cudaMemcpyDeviceToDevice, s), "export");
  if (bucket_perm) SF_CUDA_TRY(cudaMemcpyAsync(bucket_perm, p->bucket_perm, p->d * 4, cudaMemcpyDeviceToDevice, s), "export");
  return SF_OK;
}

int64_t lsp_projector_rows(lsp_projector p) { return p ? p->rows : -1; }
int32_t lsp_projector_dim(lsp_projector p) { return p ? p->d : -1; }
int32_t lsp_projector_nnz_per_row(lsp_projector p) { return p ? p->k : -1; }

sf_status lsp_projector_destroy(lsp_projector p) {
  sf::clear_error();
  if (!p) return SF_OK;
  cudaError_t e = cudaFree(p->block);
  delete p;
  return e == cudaSuccess ? SF_OK : sf::cuda_fail(e, "cudaFree(projector)");
}

size_t lsp_workspace_bytes(int64_t m, int64_t n, int32_t d) {
  if (m < 1 || n < 1 || d < 1) return 0;
  return std::max(sf::plan_compress(m, n, d).bytes, sf::decompress_bytes(n, d));
}

sf_status lsp_compress(lsp_projector P, lsp_projector Q, const void* G, sf_dtype g_dtype, int64_t m, int64_t n,
                       float* S, void* ws, size_t ws_bytes, void* stream_) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("lsp_compress");
  SF_TRY(sf::check_proj(P, "P"));
  SF_TRY(sf::check_proj(Q, "Q"));
  if (!G || !S) return fail(SF_ERR_INVALID, "G or S is NULL");
  if (P->rows != m || Q->rows != n)
    return fail(SF_ERR_INVALID, "P has %lld rows, Q %lld: need m = %lld, n = %lld", (long long)P->rows,
                (long long)Q->rows, (long long)m, (long long)n);
  if (P->d != Q->d) return fail(SF_ERR_INVALID, "P and Q differ in d (%d vs %d)", P->d, Q->d);
  if (g_dtype != SF_BF16 && g_dtype != SF_FP32) return fail(SF_ERR_INVALID, "g_dtype must be SF_BF16 or SF_FP32");
  const int d = P->d;
  const sf::CompressPlan cp = sf::plan_compress(m, n, d);
  if (!ws || ws_bytes < cp.bytes || (reinterpret_cast<uintptr_t>(ws) % 256) != 0)
    return fail(SF_ERR_INVALID, "workspace needs %zu bytes, 256-byte aligned (got %zu)", cp.bytes, ws_bytes);
  cudaStream_t s = sf::as_stream(stream_);
  char* w = static_cast<char*>(ws);
  float* rt = reinterpret_cast<float*>(w + cp.off_rt);
  float* rtp = reinterpret_cast<float*>(w + cp.off_rtp);
  float* sp = reinterpret_cast<float*>(w + cp.off_sp);
  if (g_dtype == SF_FP32)
    SF_TRY(sf::launch_gather<float>(P, static_cast<const float*>(G), n, n, cp.g1, rt, rtp, s));
  else
    SF_TRY(sf::launch_gather<__nv_bfloat16>(P, static_cast<const __nv_bfloat16*>(G), n, n, cp.g1, rt, rtp, s));
  return sf::launch_stage2(Q, rt, d, d, cp.g2, S, sp, s);
}

size_t lsp_compress_layer_workspace_bytes(int count, const int64_t* m, const int64_t* n, int32_t d) {
  if (count < 1 || !m || !n || d < 1) return 0;
  size_t total = 0;
  for (int i = 0; i < count; ++i) {
    if (m[i] < 1 || n[i] < 1) return 0;
    total += sf::align_up(sf::plan_compress(m[i], n[i], d).bytes, 256);
  }
  return total;
}

sf_status lsp_compress_layer(int count, const lsp_projector* P, const lsp_projector* Q, const void* const* G,
                             const int32_t* g_dtype, const int64_t* m, const int64_t* n, float* const* S, void* ws,
                             size_t ws_bytes, void* stream_) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("lsp_compress_layer");
  if (count < 1 || !P || !Q || !G || !g_dtype || !m || !n || !S)
    return fail(SF_ERR_INVALID, "need count >= 1 and non-NULL arrays");
  int d = 0;
  for (int i = 0; i < count; ++i) {
    SF_TRY(sf::check_proj(P[i], "P[i]"));
    SF_TRY(sf::check_proj(Q[i], "Q[i]"));
    if (!G[i] || !S[i]) return fail(SF_ERR_INVALID, "matrix %d: G or S is NULL", i);
    if (P[i]->rows != m[i] || Q[i]->rows != n[i])
      return fail(SF_ERR_INVALID, "matrix %d: P has %lld rows, Q %lld: need m = %lld, n = %lld", i,
                  (long long)P[i]->rows, (long long)Q[i]->rows, (long long)m[i], (long long)n[i]);
    if (P[i]->d != Q[i]->d || (i > 0 && P[i]->d != d))
      return fail(SF_ERR_INVALID, "matrix %d: every projector of the layer needs the same d", i);
    d = P[i]->d;
    if (g_dtype[i] != SF_BF16 && g_dtype[i] != SF_FP32)
      return fail(SF_ERR_INVALID, "matrix %d: g_dtype must be SF_BF16 or SF_FP32", i);
  }
  const size_t need = lsp_compress_layer_workspace_bytes(count, m, n, d);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % 256) != 0)
    return fail(SF_ERR_INVALID, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  cudaStream_t s = sf::as_stream(stream_);
  std::vector<sf::CompressPlan> cp(count);
  std::vector<float*> rt(count), rtp(count), sp(count);
  std::vector<int64_t> ld(count), dd(count, d);
  char* w = static_cast<char*>(ws);
  for (int i = 0; i < count; ++i) {
    cp[i] = sf::plan_compress(m[i], n[i], d);
    rt[i] = reinterpret_cast<float*>(w + cp[i].off_rt);
    rtp[i] = reinterpret_cast<float*>(w + cp[i].off_rtp);
    sp[i] = reinterpret_cast<float*>(w + cp[i].off_sp);
    ld[i] = n[i];
    w += sf::align_up(cp[i].bytes, 256);
  }
  // stage 1, one launch per element type of G
  for (const int32_t dt : {(int32_t)SF_FP32, (int32_t)SF_BF16}) {
    std::vector<const lsp_projector_s*> a;
    std::vector<const void*> b;
    std::vector<int64_t> ldb, nc;
    std::vector<sf::GatherPlan> pl;
    std::vector<float*> yf, yp;
    for (int i = 0; i < count; ++i) {
      if (g_dtype[i] != dt) continue;
      a.push_back(P[i]);
      b.push_back(G[i]);
      ldb.push_back(n[i]);
      nc.push_back(n[i]);
      pl.push_back(cp[i].g1);
      yf.push_back(rt[i]);
      yp.push_back(rtp[i]);
    }
    if (a.empty()) continue;
    if (dt == SF_FP32)
      SF_TRY(sf::launch_gather_multi<float>((int)a.size(), a.data(), reinterpret_cast<const float* const*>(b.data()),
                                            ldb.data(), nc.data(), pl.data(), yf.data(), yp.data(), s));
    else
      SF_TRY(sf::launch_gather_multi<__nv_bfloat16>((int)a.size(), a.data(),
                                                    reinterpret_cast<const __nv_bfloat16* const*>(b.data()),
                                                    ldb.data(), nc.data(), pl.data(), yf.data(), yp.data(), s));
  }
  // stage 2 for every matrix
  std::vector<const lsp_projector_s*> q(Q, Q + count);
  std::vector<const float*> rtc(rt.begin(), rt.end());
  std::vector<sf::GatherPlan> p2(count);
  for (int i = 0; i < count; ++i) p2[i] = cp[i].g2;
  return sf::launch_stage2_multi(count, q.data(), rtc.data(), dd.data(), dd.data(), p2.data(), S, sp.data(), s);
}

}  // extern "C"

// ----------------------------------------------------------------------------
// lsp_compress without a caller workspace
// ----------------------------------------------------------------------------
// Some callers cannot hand the library a device workspace: code that runs
// under a framework whose caching allocator owns the device memory pool (a
// raw cudaMalloc there competes with, or fails against, that pool), code in
// a latency-critical loop where cudaMalloc's implicit device-wide
// synchronisation is not acceptable, and thin bindings that have no
// allocator of their own.  For them the compress intermediate lives in this
// fixed array instead.  It is part of the library image: every GPU that
// loads the library holds it until the process exits.
namespace sf {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SF_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, never a device address, so
// it is never passed to a kernel.  The address is looked up on every call
// (a lookup costs little next to a compress): a cached one would go stale
// when the device is reset and the library's device code loaded anew.
sf_status noalloc_scratch(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
  *out = p;
  return SF_OK;
}

}  // namespace
}  // namespace sf

extern "C" {

sf_status lsp_compress_noalloc(lsp_projector P, lsp_projector Q, const void* G, sf_dtype g_dtype, int64_t m, int64_t n,
                               float* S, void* stream) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("lsp_compress_noalloc");
  SF_TRY(sf::check_proj(P, "P"));
  SF_TRY(sf::check_proj(Q, "Q"));
  if (P->rows != m || Q->rows != n)
    return fail(SF_ERR_INVALID, "P has %lld rows, Q %lld: need m = %lld, n = %lld", (long long)P->rows,
                (long long)Q->rows, (long long)m, (long long)n);
  if (P->d != Q->d) return fail(SF_ERR_INVALID, "P and Q differ in d (%d vs %d)", P->d, Q->d);
  const size_t need = sf::plan_compress(m, n, P->d).bytes;
  if (need > (size_t)SF_NOALLOC_SCRATCH_BYTES)
    return fail(SF_ERR_UNSUPPORTED,
                "lsp_compress_noalloc: this shape needs %zu bytes of scratch, above the fixed %zu bytes; "
                "use lsp_compress with a workspace",
                need, (size_t)SF_NOALLOC_SCRATCH_BYTES);
  void* ws = nullptr;
  SF_TRY(sf::noalloc_scratch(&ws));
  // Everything the compress writes into the scratch is written before it is
  // read, so nothing needs clearing between calls.
  return lsp_compress(P, Q, G, g_dtype, m, n, S, ws, (size_t)SF_NOALLOC_SCRATCH_BYTES, stream);
}

sf_status lsp_decompress_apply(lsp_projector P, lsp_projector Q, const float* dS, void* W, sf_dtype w_dtype,
                               void* w_bf16_mirror, int64_t m, int64_t n, void* ws, size_t ws_bytes, void* stream_) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("lsp_decompress_apply");
  SF_TRY(sf::check_proj(P, "P"));
  SF_TRY(sf::check_proj(Q, "Q"));
  if (!dS || !W) return fail(SF_ERR_INVALID, "dS or W is NULL");
  if (P->rows != m || Q->rows != n)
    return fail(SF_ERR_INVALID, "P has %lld rows, Q %lld: need m = %lld, n = %lld", (long long)P->rows,
                (long long)Q->rows, (long long)m, (long long)n);
  if (P->d != Q->d) return fail(SF_ERR_INVALID, "P and Q differ in d (%d vs %d)", P->d, Q->d);
  if (w_dtype != SF_BF16 && w_dtype != SF_FP32) return fail(SF_ERR_INVALID, "w_dtype must be SF_BF16 or SF_FP32");
  if (w_bf16_mirror && w_dtype != SF_FP32) return fail(SF_ERR_INVALID, "a bf16 mirror needs an fp32 W");
  const int d = P->d;
  const size_t need = sf::decompress_bytes(n, d);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % 256) != 0)
    return fail(SF_ERR_INVALID, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  cudaStream_t s = sf::as_stream(stream_);
  float* V = static_cast<float*>(ws);
  const int nsm = sf::sm_count();
  uint16_t* mirror = static_cast<uint16_t*>(w_bf16_mirror);
  if (d <= sf::kMaxFastD && P->k <= 32 && Q->k <= 32) {
    const int n_ab = (int)ceil_div(d, sf::kVRows);
    // one wave: about one CTA per SM, each with a column range that is a
    // multiple of the 8-column group
    const int64_t n_groups = ceil_div<int64_t>(n, sf::kVGroup);
    const int64_t gy = std::max<int64_t>(1, std::min<int64_t>(n_groups, nsm / n_ab));
    const int64_t cols_per_cta = ceil_div<int64_t>(n_groups, gy) * sf::kVGroup;
    const int64_t gy_used = ceil_div<int64_t>(n, cols_per_cta);
    float* dSt = reinterpret_cast<float*>(static_cast<char*>(ws) + sf::align_up((size_t)d * n * 4, 256));
    const bool rows_form = Q->k == 8 && d % 64 == 0 && n % sf::kVGroup == 0 &&
                           (reinterpret_cast<uintptr_t>(V) % 16) == 0;
    if (rows_form) {
      // dS^T once (1 MB at d = 512), then V by row gathers of it
      SF_CUDA_TRY(sf::launch_pdl(sf::k_transpose_dd, dim3((unsigned)ceil_div(d, 32), (unsigned)ceil_div(d, 32)),
                                 dim3(32, 8), 0, s, dS, d, dSt),
                  "launch k_transpose_dd");
      const int64_t n_groups = n / sf::kVGroup;
      const int64_t gx = std::max<int64_t>(1, ceil_div<int64_t>(n_groups, (int64_t)sf::kVrWarps * sf::kVrGroupsPerWarp));
      SF_CUDA_TRY(sf::launch_pdl(sf::k_v_rows, dim3((unsigned)gx, (unsigned)(d / 64)), dim3(32 * sf::kVrWarps), 0, s,
                                 dSt, d, Q->ell_idx, Q->ell_val, n, V),
                  "launch k_v_rows");
    } else if (Q->k <= sf::kVMaxK) {
      const size_t smem_v = sf::v_smem_bytes(d);
      SF_TRY(sf::allow_dynamic_smem(reinterpret_cast<const void*>(&sf::k_v), sf::v_smem_bytes(sf::kMaxFastD)));
      SF_CUDA_TRY(sf::launch_pdl(sf::k_v, dim3((unsigned)n_ab, (unsigned)gy_used), dim3(32 * sf::kVWarps), smem_v, s,
                                 dS, d, Q->ell_idx, Q->ell_val, Q->k, n, V, cols_per_cta),
                  "launch k_v");
    } else {
      const int64_t nv = (int64_t)d * n;
      sf::k_v_generic<<<(unsigned)ceil_div<int64_t>(nv, 256), 256, 0, s>>>(dS, d, Q->ell_idx, Q->ell_val, Q->k, n, V);
      SF_TRY(sf::check_launch("k_v_generic"));
    }

    const size_t smem_a = (size_t)d * sf::kApplyCols * 4 + 16 * 32 * 8;
    const int64_t n_jb = ceil_div<int64_t>(n, sf::kApplyCols);
    const int64_t total = n_jb * m;
    const bool bf16w = w_dtype == SF_BF16;
    auto kern = bf16w ? sf::k_apply<true> : sf::k_apply<false>;
    SF_TRY(sf::allow_dynamic_smem(reinterpret_cast<const void*>(kern),
                                  (size_t)sf::kMaxFastD * sf::kApplyCols * 4 + 16 * 32 * 8));
    int occ = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 512, smem_a);
    occ = std::max(1, occ);
    const int64_t grid = std::min<int64_t>((int64_t)nsm * occ, ceil_div<int64_t>(total, 16));
    const int64_t ipc = ceil_div<int64_t>(total, grid);
    const size_t wb = bf16w ? 2 : 4;
    const int vec_ok = (n % 2 == 0) && (reinterpret_cast<uintptr_t>(W) % (2 * wb) == 0) &&
                       (!mirror || reinterpret_cast<uintptr_t>(mirror) % 4 == 0);
    const size_t wes = bf16w ? 2 : 4;
    if (sf::tma_ok(W, n, wes)) {
      sf::ApplyArgs A;
      A.V = V;
      A.pidx = P->ell_idx;
      A.pval = P->ell_val;
      A.W = W;
      A.mirror = mirror;
      A.n = n;
      A.m = m;
      A.n_rt = ceil_div<int64_t>(m, sf::kApplyRows);
      A.total = n_jb * A.n_rt;
      A.d = d;
      A.k = P->k;
      A.tile_bytes = sf::kApplyRows * sf::kApplyCols * (int)wes;
      A.ent_stride = (int)sf::align_up((size_t)sf::kApplyRows * P->k * 4, 128);
      A.stage_stride = (int)sf::align_up((size_t)A.tile_bytes + 2 * A.ent_stride, 1024);
      A.vs_bytes = (int)sf::align_up((size_t)d * sf::kApplyCols * 4, 1024);
      const size_t fixed = (size_t)A.vs_bytes + 2 * sf::kApplyMaxStages * 8 + 16 + 1024;
      A.stages = (int)std::min<size_t>(sf::kApplyMaxStages, (220 * 1024 - fixed) / A.stage_stride);
      if (A.stages >= 2) {
        A.vec_ok = vec_ok;
        A.v_vec = (n % 4 == 0) && (reinterpret_cast<uintptr_t>(V) % 16 == 0) ? 1 : 0;
        const int64_t grid2 = std::min<int64_t>(nsm, A.total);
        A.per_cta = ceil_div<int64_t>(A.total, grid2);
        const size_t smem2 = fixed + (size_t)A.stages * A.stage_stride;
        CUtensorMap wmap;
        cuuint64_t dims[2] = {(cuuint64_t)n, (cuuint64_t)m};
        cuuint64_t strides[1] = {(cuuint64_t)(n * (int64_t)wes)};
        cuuint32_t box[2] = {(cuuint32_t)sf::kApplyCols, (cuuint32_t)sf::kApplyRows};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = sf::tensor_map_encoder()(&wmap, bf16w ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                                              2, W, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(SF_ERR_CUDA, "cuTensorMapEncodeTiled(W) failed (%d)", (int)r);
        auto kt = bf16w ? sf::k_apply_tma<true> : sf::k_apply_tma<false>;
        SF_TRY(sf::allow_dynamic_smem(reinterpret_cast<const void*>(kt), 220 * 1024));
        SF_CUDA_TRY(sf::launch_pdl(kt, dim3((unsigned)ceil_div<int64_t>(A.total, A.per_cta)),
                                   dim3(32 * (sf::kApplyConsumerWarps + 1)), smem2, s, wmap, A),
                    "launch k_apply_tma");
        return SF_OK;
      }
    }
    const int R = std::min(sf::kApplyMaxR, 32 / P->k);
    kern<<<(unsigned)ceil_div<int64_t>(total, ipc), 512, smem_a, s>>>(V, d, n, m, P->ell_idx, P->ell_val, P->k, R, W,
                                                                       mirror, total, ipc, vec_ok);
    return sf::check_launch("k_apply");
  }
  const int64_t nv = (int64_t)d * n;
  sf::k_v_generic<<<(unsigned)ceil_div<int64_t>(nv, 256), 256, 0, s>>>(dS, d, Q->ell_idx, Q->ell_val, Q->k, n, V);
  SF_TRY(sf::check_launch("k_v_generic"));
  const int64_t nw = m * n;
  if (w_dtype == SF_BF16)
    sf::k_apply_generic<true><<<(unsigned)ceil_div<int64_t>(nw, 256), 256, 0, s>>>(V, n, m, P->ell_idx, P->ell_val,
                                                                                   P->k, W, nullptr);
  else
    sf::k_apply_generic<false><<<(unsigned)ceil_div<int64_t>(nw, 256), 256, 0, s>>>(V, n, m, P->ell_idx, P->ell_val,
                                                                                    P->k, W, mirror);
  return sf::check_launch("k_apply_generic");
}

}  // extern "C"

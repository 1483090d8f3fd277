// Declarations shared by the projector translation units: the projector
// handle (lsp.cu builds it; lsp_fit.cu updates its values) and the gather
// machinery of the compress stages, which the fit step reuses.
#pragma once

#include <cuda_bf16.h>

#include "common.h"

// ----------------------------------------------------------------------------
// Projector handle
// ----------------------------------------------------------------------------
struct lsp_projector_s {
  int device = 0;
  int64_t rows = 0;
  int32_t d = 0, k = 0, dp = 0, n_win = 0;
  int32_t* ell_idx = nullptr;   // [rows*k], out-of-range ids replaced by (0, 0.0f)
  float* ell_val = nullptr;
  int32_t* col_ptr = nullptr;   // [d+1]
  int32_t* row_idx = nullptr;   // [rows*k]
  float* csc_val = nullptr;
  int32_t* bucket_perm = nullptr;  // [d]
  int32_t* wptr = nullptr;      // [n_win*dp + 1]: start of (window, a) in went
  int2* went = nullptr;         // [rows*k]: (row, value bits), sorted by (window, a, row)
  int2* gdesc = nullptr;        // [n_ar][n_win]: (first entry rounded down to even, bytes) of a CTA's slice
  int32_t a_rng = 0, n_ar = 0;  // outputs per gather CTA (8 x warps) and number of such ranges
  int32_t max_slice_bytes = 0;  // largest gdesc byte count
  int32_t* ell2csc = nullptr;   // [rows*k]: position of ELL entry e in the CSC arrays (-1: id out of range)
  int32_t* ell2went = nullptr;  // [rows*k]: position of ELL entry e in went (-1: id out of range)
  bool bad_ids = false;         // some id was out of range at creation
  int32_t* wcnt = nullptr;      // [n_win*dp] scratch of the build
  int32_t* csc_off = nullptr;   // [n_win*dp] scratch of the build
  int32_t* totals = nullptr;    // [d] scratch of the build
  int32_t* err = nullptr;       // [2]: error bits, largest slice bytes
  void* block = nullptr;
};

namespace sf {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch geometry of one gather (pure function of the sizes).
struct GatherPlan {
  int warps, n_ar, n_cb, n_win, splits, win_per_split;
  // tail_splits > 1: a 1D grid, column blocks [0, cb_main) whole, the rest
  // split tail_splits ways over tail_wps windows each
  int cb_main, tail_splits, tail_wps;
  size_t partial_bytes;   // partials either form needs
};

// The two gathers of lsp_compress and the workspace they use.
struct CompressPlan {
  GatherPlan g1, g2;
  bool stage2_rows;     // stage 2 as the row gather straight from L2 (no partials)
  size_t off_rt, off_rtp, off_sp, bytes;
};

GatherPlan plan_gather(int64_t rows, int64_t ncols, int d);
CompressPlan plan_compress(int64_t m, int64_t n, int d);

// Y^T = (A^T B)^T for projector A (rows = rows of B) and B [rows][ldb] of
// type TB (float or __nv_bfloat16), ncols columns; yt_final [ncols][d],
// yt_partial the split partials the plan needs.  Enqueued on `stream`.
template <typename TB>
sf_status launch_gather(const lsp_projector_s* Aproj, const TB* B, int64_t ldb, int64_t ncols, const GatherPlan& p,
                        float* yt_final, float* yt_partial, cudaStream_t stream);

// SF_ERR_INVALID unless p is a projector built on the current device.
// Second compress stage, Y^T = (A^T B)^T for a small L2-resident fp32 B:
// a row gather straight from L2 when B's rows are 16-byte aligned, else
// launch_gather (plan p, partials yt_partial).
sf_status launch_stage2(const lsp_projector_s* Aproj, const float* B, int64_t ldb, int64_t ncols, const GatherPlan& p,
                        float* yt_final, float* yt_partial, cudaStream_t stream);

sf_status check_proj(const lsp_projector_s* p, const char* name);

}  // namespace sf

// Internal helpers shared by the library's translation units: status and
// error-message plumbing, argument checks, small integer utilities.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <string>

#include "sfopt.h"

namespace sf {

// NVTX range around one ABI call, so profiler timelines show library calls
// by name (header-only NVTX; a no-op unless a tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Records a message for sf_last_error() (thread-local) and returns `st`.
sf_status fail(sf_status st, const char* fmt, ...);

// Clears the calling thread's last error message.
void clear_error();

// Maps a CUDA error to SF_ERR_CUDA with a message naming `what`.
sf_status cuda_fail(cudaError_t e, const char* what);

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

template <typename T>
constexpr T ceil_div(T a, T b) { return (a + b - 1) / b; }

// Number of SMs of the current device (cached per device).
int sm_count();

// Lets kernel `func` use up to `bytes` of dynamic shared memory on the
// current device (cudaFuncSetAttribute once per device, kernel and size;
// thread-safe).
sf_status allow_dynamic_smem(const void* func, size_t bytes);

// cuTensorMapEncodeTiled from the driver (looked up once), or null.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// True when `p` points into device memory of the current device.  Every
// tensor map (TMA descriptor) this library encodes addresses such memory
// only; operands elsewhere (pinned host memory, a peer GPU's memory) take a
// path with plain loads or are rejected.
bool on_current_device(const void* p);

// Default bound for host waits, in milliseconds (SF_TIMEOUT_MS or 600 s).
int64_t default_timeout_ms();

// Polls `ev` (or a stream when ev is null) until it completes or the bound
// runs out.  Returns SF_OK, SF_ERR_TIMEOUT or SF_ERR_CUDA.
sf_status bounded_wait_event(cudaEvent_t ev, int64_t timeout_ms, const char* what);
sf_status bounded_wait_stream(cudaStream_t s, int64_t timeout_ms, const char* what);

// Checks for a pending launch error after enqueueing kernels.
inline sf_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SF_OK : cuda_fail(e, what);
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel in the stream drains; it must call
// griddepcontrol.wait before touching memory that kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// fp32 constants of one AdamW step, derived in double and rounded once.
struct AdamConsts {
  float beta1, one_minus_beta1;
  float beta2, one_minus_beta2;
  float decay;          // 1 - lr * weight_decay
  float step_size;      // lr / (1 - beta1^t)
  float sqrt_bc2;       // sqrt(1 - beta2^t)
  float inv_sqrt_bc2;   // 1 / sqrt(1 - beta2^t), rounded once from double
  float eps;
};

// Reads and clears the device-side error word that bounded waits and index
// checks in the kernels set (0 = none; bit 1 = a wait ran out; bit 2 = an
// out-of-range index was skipped).
int read_and_clear_device_error();
int read_and_clear_device_error_adamw();
int read_and_clear_device_error_gemm();
int read_and_clear_device_error_lce();

// C = alpha A B^T (+ C) on the tensor cores (tc_gemm.cu): A bf16 [M][lda]
// row-major (K-major) or, with a_mn, [K][lda] (MN-major: A^T stored);
// B likewise [N][ldb] or, with b_mn, [K][ldb]; C fp32 [M][ldc].  With
// row_stats (float2 [M][ceil(N / 256)]) the epilogue also writes, per row and
// 256-column tile, the maximum of the row's values and the sum of
// exp(value - maximum).
constexpr int kTcTileN = 256;
sf_status tc_gemm(const void* A, bool a_mn, const void* B, bool b_mn, float* C, int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc, float alpha, bool accumulate, cudaStream_t s,
                  float2* row_stats = nullptr);

sf_status make_adam_consts(const sf_adamw_hparams* hp, int64_t step, bool with_decay,
                           AdamConsts* out);

// The compressed AdamW step on the host cores for elements [b, e) of fp32
// S, m, v -> dS (host_adamw.cpp): bitwise the device kernel's results.
void host_adamw_compressed(const float* S, float* m, float* v, float* dS, int64_t b, int64_t e,
                           const AdamConsts& c);

// Cores this process may run on (its CPU affinity set), at least 1.
int usable_cores();

}  // namespace sf

#define SF_TRY(expr)                      \
  do {                                    \
    sf_status _st = (expr);               \
    if (_st != SF_OK) return _st;         \
  } while (0)

#define SF_CUDA_TRY(expr, what)                       \
  do {                                                \
    cudaError_t _e = (expr);                          \
    if (_e != cudaSuccess) return sf::cuda_fail(_e, what); \
  } while (0)

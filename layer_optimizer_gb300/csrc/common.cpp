// Status plumbing, bounded host waits and AdamW constant derivation.
#include "common.h"

#include <map>
#include <mutex>
#include <utility>

#include <sched.h>

#include <chrono>
#include <cmath>
#include <cstdlib>
#include <thread>

namespace sf {

namespace {
thread_local std::string g_last_error;
}

sf_status fail(sf_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

void clear_error() { g_last_error.clear(); }

sf_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SF_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

int sm_count() {
  static thread_local int cached_dev = -1, cached_sms = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev != cached_dev) {
    int sms = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cached_dev = dev;
    cached_sms = sms > 0 ? sms : 1;
  }
  return cached_sms;
}

bool on_current_device(const void* p) {
  if (!p) return false;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

int usable_cores() {
  cpu_set_t set;
  CPU_ZERO(&set);
  if (sched_getaffinity(0, sizeof set, &set) == 0) {
    const int n = CPU_COUNT(&set);
    if (n > 0) return n;
  }
  const unsigned h = std::thread::hardware_concurrency();
  return h > 0 ? (int)h : 1;
}

int64_t default_timeout_ms() {
  const char* s = std::getenv("SF_TIMEOUT_MS");
  if (s && *s) {
    long long v = std::atoll(s);
    if (v > 0) return v;
  }
  return 600000;
}

namespace {
template <typename Query>
sf_status poll(Query q, int64_t timeout_ms, const char* what) {
  if (timeout_ms <= 0) timeout_ms = default_timeout_ms();
  auto t0 = std::chrono::steady_clock::now();
  int64_t sleep_us = 0;
  for (;;) {
    cudaError_t e = q();
    if (e == cudaSuccess) return SF_OK;
    if (e != cudaErrorNotReady) return cuda_fail(e, what);
    auto el = std::chrono::duration_cast<std::chrono::milliseconds>(
                  std::chrono::steady_clock::now() - t0).count();
    if (el >= timeout_ms)
      return fail(SF_ERR_TIMEOUT, "%s: still running after %lld ms", what, (long long)el);
    if (sleep_us > 0) std::this_thread::sleep_for(std::chrono::microseconds(sleep_us));
    sleep_us = sleep_us == 0 ? 1 : (sleep_us < 200 ? sleep_us * 2 : 200);
  }
}
}  // namespace

sf_status bounded_wait_event(cudaEvent_t ev, int64_t timeout_ms, const char* what) {
  return poll([&] { return cudaEventQuery(ev); }, timeout_ms, what);
}

sf_status bounded_wait_stream(cudaStream_t s, int64_t timeout_ms, const char* what) {
  return poll([&] { return cudaStreamQuery(s); }, timeout_ms, what);
}

sf_status make_adam_consts(const sf_adamw_hparams* hp, int64_t step, bool with_decay,
                           AdamConsts* out) {
  if (!hp) return fail(SF_ERR_INVALID, "hyper-parameters are NULL");
  if (step < 1) return fail(SF_ERR_INVALID, "step must be >= 1 (got %lld)", (long long)step);
  const double v[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
  for (double x : v)
    if (!std::isfinite(x)) return fail(SF_ERR_INVALID, "non-finite hyper-parameter");
  if (!(hp->beta1 >= 0.0 && hp->beta1 < 1.0) || !(hp->beta2 >= 0.0 && hp->beta2 < 1.0))
    return fail(SF_ERR_INVALID, "betas must lie in [0, 1)");
  const double t = static_cast<double>(step);
  const double bc1 = 1.0 - std::pow(hp->beta1, t);
  const double bc2 = 1.0 - std::pow(hp->beta2, t);
  out->beta1 = static_cast<float>(hp->beta1);
  out->one_minus_beta1 = static_cast<float>(1.0 - hp->beta1);
  out->beta2 = static_cast<float>(hp->beta2);
  out->one_minus_beta2 = static_cast<float>(1.0 - hp->beta2);
  out->decay = static_cast<float>(with_decay ? 1.0 - hp->lr * hp->weight_decay : 1.0);
  out->step_size = static_cast<float>(hp->lr / bc1);
  out->sqrt_bc2 = static_cast<float>(std::sqrt(bc2));
  out->inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
  out->eps = static_cast<float>(hp->eps);
  return SF_OK;
}

sf_status allow_dynamic_smem(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = done[{dev, func}];
  if (have >= bytes) return SF_OK;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
  have = bytes;
  return SF_OK;
}

}  // namespace sf

extern "C" {

const char* sf_last_error(void) { return sf::g_last_error.c_str(); }

const char* sf_version(void) { return "0.1.0"; }

sf_status sf_sync_status(void* stream) {
  sf::clear_error();
  SF_TRY(sf::bounded_wait_stream(sf::as_stream(stream), 0, "sf_sync_status"));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return sf::cuda_fail(e, "sf_sync_status");
  const int dev_err = sf::read_and_clear_device_error() | sf::read_and_clear_device_error_adamw() |
                      sf::read_and_clear_device_error_gemm() | sf::read_and_clear_device_error_lce();
  if (dev_err & 1) return sf::fail(SF_ERR_TIMEOUT, "a kernel wait ran out of its bound (device error word %d)", dev_err);
  if (dev_err & 2) return sf::fail(SF_ERR_INVALID, "a kernel skipped an out-of-range index (device error word %d)", dev_err);
  return SF_OK;
}

}  // extern "C"

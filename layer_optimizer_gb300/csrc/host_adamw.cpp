// The AdamW layer step on the host CPU cores, multi-threaded.
//
// SlideFormer ("An Efficient Heterogeneous Co-Design for Fine-Tuning on a
// Single GPU", technical summary section 2.A) runs the optimizer step of a
// layer on CPU threads over flattened fp32 states in host memory while the
// GPU computes the next layer.  This is that update, as a comparison point
// for the on-device kernels: the same arithmetic, element for element, as
// adamw.cu (the file is compiled without floating-point contraction and uses
// explicit fused multiply-adds where the kernel does), so on IEEE hardware
// it produces the same bits as the GPU.
//
// Threads split the layer's elements into contiguous ranges (across tensor
// boundaries); every element is touched by exactly one thread.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "common.h"

namespace {

// Round-to-nearest-even of an fp32 value to bfloat16 (the top 16 bits),
// from the binary32 layout: add half an ulp of the kept part, plus one if
// the kept part is odd (ties to even); NaN stays a quiet NaN.
uint16_t bf16_rne(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

float bf16_to_f32(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

void update_range(const sf_tensor& t, int64_t b, int64_t e, const sf::AdamConsts& c) {
  const uint16_t* g = static_cast<const uint16_t*>(t.grad);
  uint16_t* w = static_cast<uint16_t*>(t.weight);
  float* P = t.master;
  float* M = t.exp_avg;
  float* V = t.exp_avg_sq;
  for (int64_t i = b; i < e; ++i) {
    const float gi = bf16_to_f32(g[i]);
    const float m = std::fmaf(c.beta1, M[i], c.one_minus_beta1 * gi);
    const float v = std::fmaf(c.beta2, V[i], c.one_minus_beta2 * (gi * gi));
    const float denom = std::fmaf(std::sqrt(v), c.inv_sqrt_bc2, c.eps);
    const float p = std::fmaf(-c.step_size, m / denom, P[i] * c.decay);
    M[i] = m;
    V[i] = v;
    P[i] = p;
    if (w) w[i] = bf16_rne(p);
  }
}

}  // namespace

namespace sf {

// The compressed AdamW step (adamw.cu, adamw_compressed_kernel) on elements
// [b, e) of fp32 S, m, v -> dS on the host: the same operations in the same
// order, so the same bits.
void host_adamw_compressed(const float* S, float* m, float* v, float* dS, int64_t b, int64_t e,
                           const AdamConsts& c) {
  for (int64_t i = b; i < e; ++i) {
    const float g = S[i];
    const float mm = std::fmaf(c.beta1, m[i], c.one_minus_beta1 * g);
    const float vv = std::fmaf(c.beta2, v[i], c.one_minus_beta2 * (g * g));
    const float denom = std::fmaf(std::sqrt(vv), c.inv_sqrt_bc2, c.eps);
    m[i] = mm;
    v[i] = vv;
    dS[i] = c.step_size * (mm / denom);
  }
}

}  // namespace sf

extern "C" {

sf_status sf_adamw_host_step(const sf_tensor* tensors, int n_tensors, const sf_adamw_hparams* hp, int64_t step,
                             int n_threads) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("sf_adamw_host_step");
  if (n_tensors < 0) return sf::fail(SF_ERR_INVALID, "n_tensors < 0");
  if (n_tensors > 0 && !tensors) return sf::fail(SF_ERR_INVALID, "tensors is NULL");
  sf::AdamConsts c;
  SF_TRY(sf::make_adam_consts(hp, step, true, &c));
  int64_t total = 0;
  std::vector<int64_t> start(n_tensors + 1, 0);
  for (int i = 0; i < n_tensors; ++i) {
    const sf_tensor& t = tensors[i];
    if (t.numel < 0) return sf::fail(SF_ERR_INVALID, "tensor %d: numel < 0", i);
    if (t.numel > 0 && (!t.grad || !t.master || !t.exp_avg || !t.exp_avg_sq))
      return sf::fail(SF_ERR_INVALID, "tensor %d: grad/master/exp_avg/exp_avg_sq must be non-NULL", i);
    start[i] = total;
    total += t.numel;
  }
  start[n_tensors] = total;
  if (total == 0) return SF_OK;
  int nt = n_threads > 0 ? n_threads : sf::usable_cores();
  nt = (int)std::min<int64_t>(nt, std::max<int64_t>(1, total / 65536));

  // thread k owns global elements [k*total/nt, (k+1)*total/nt)
  auto work = [&](int k) {
    const int64_t b = total * k / nt, e = total * (k + 1) / nt;
    for (int i = 0; i < n_tensors; ++i) {
      const int64_t tb = std::max(b, start[i]), te = std::min(e, start[i + 1]);
      if (tb < te) update_range(tensors[i], tb - start[i], te - start[i], c);
    }
  };
  std::vector<std::thread> pool;
  pool.reserve(nt - 1);
  try {
    for (int k = 1; k < nt; ++k) pool.emplace_back(work, k);
  } catch (...) {
    for (auto& th : pool) th.join();
    return sf::fail(SF_ERR_OOM, "could not start %d host threads", nt);
  }
  work(0);
  for (auto& th : pool) th.join();
  return SF_OK;
}

}  // extern "C"

// Layer-sliding window: streams layers between pinned host memory and a
// fixed set of pre-allocated device slots on three CUDA streams, with the
// fused AdamW update in between.
//
// SlideFormer ("An Efficient Heterogeneous Co-Design for Fine-Tuning on a
// Single GPU", technical summary section 2.A) keeps only a small active
// window of layers on the GPU and overlaps computation, host<->device
// transfer and the optimizer update of neighbouring layers; section 2.B
// pre-allocates a fixed queue of GPU cache units, each holding one layer,
// so nothing is allocated while training runs.  This engine is that
// window for the update step: a visit copies one layer into a free slot
// (h2d stream), updates it (compute stream), and copies it back (d2h
// stream).  Visits to different slots run concurrently, so the copy
// engines in both directions and the HBM-bound kernel overlap.  Inside a
// visit the layer moves in groups of consecutive tensors (at least
// kGroupParams parameters each, or the rest of the layer): a group's update
// starts as soon as that group has arrived, its write-back as soon as it is
// updated, and the next visit to the slot may overwrite a tensor as soon as
// that tensor's write-back has ended.  Copies go per array of a group, and
// tensors whose host and slot arrays both follow one another in memory
// move as one copy (a layer kept as flat per-array buffers, as flattened
// optimizer states are, costs one copy per array).  An array of a layer that
// already lives in this device's memory (say fp32 master weights and
// moments kept resident in HBM while gradients arrive from and bf16 weights
// return to the host) is updated in place and never copied: the window then
// moves only the host-resident arrays.  It does no arithmetic of its own;
// dependencies are CUDA events only, and the host never blocks while
// enqueueing.
#include <algorithm>
#include <new>
#include <vector>

#include "common.h"

namespace sf {
sf_status adamw_layer_step_impl(const sf_tensor* tensors, int n_tensors, const sf_adamw_hparams* hp,
                                int64_t step, cudaStream_t stream);
}

struct sf_window_s {
  int device = 0;
  int n_slots = 0;
  int n_tensors = 0;
  std::vector<std::vector<sf_tensor>> slots;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  // per (slot, tensor): events of the group that starts at that tensor:
  // its copies landed / its update ended
  std::vector<cudaEvent_t> ev_in, ev_done;
  // per (slot, tensor): the write-back of the group that last held that
  // tensor of the slot has ended (recorded for every tensor of the group),
  // and the number of that group's recording (0 = never used), so a group
  // waits once per distinct earlier group
  std::vector<cudaEvent_t> ev_free;
  std::vector<int64_t> free_gen;
  int64_t gen = 0;
  std::vector<cudaEvent_t> ev_layer;   // write-back of a host layer has landed
  std::vector<bool> layer_pending;
  int64_t visits = 0;                  // running visit counter (slot rotation)
};

namespace {

constexpr int64_t kGroupParams = int64_t(64) << 20;

// Test hook: the n-th copy enqueue (1-based) fails once; 0 = off.
int64_t g_fail_copy_at = 0;
int64_t g_copy_count = 0;

sf_status copy_async(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s,
                     const char* what) {
  if (bytes == 0) return SF_OK;
  ++g_copy_count;
  if (g_fail_copy_at > 0 && g_copy_count == g_fail_copy_at) {
    g_fail_copy_at = 0;
    return sf::fail(SF_ERR_CUDA, "%s: injected copy failure", what);
  }
  cudaError_t e = cudaMemcpyAsync(dst, src, bytes, kind, s);
  return e == cudaSuccess ? SF_OK : sf::cuda_fail(e, what);
}

// The arrays of a tensor that move over the link.
enum Part { kGrad, kMaster, kExpAvg, kExpAvgSq, kWeight };

inline void* part_ptr(const sf_tensor& t, Part k) {
  switch (k) {
    case kGrad: return const_cast<void*>(t.grad);
    case kMaster: return t.master;
    case kExpAvg: return t.exp_avg;
    case kExpAvgSq: return t.exp_avg_sq;
    default: return t.weight;
  }
}
inline size_t part_bytes(Part k) { return (k == kGrad || k == kWeight) ? 2 : 4; }

// Copies array `k` of tensors [t0, t1) between the host layer and the slot.
// Tensors whose host arrays and slot arrays both follow one another in
// memory (a layer kept as flat per-array buffers, as flattened optimizer
// states are) move as one copy: one descriptor instead of one per tensor.
// A tensor without that array (a NULL weight) or whose array is resident in
// device memory (bit k of resident[t]) ends a run and is skipped.
sf_status copy_runs(const sf_host_layer& L, const std::vector<sf_tensor>& slot, const uint8_t* resident, int t0,
                    int t1, Part k, cudaMemcpyKind kind, cudaStream_t s, const char* what) {
  const size_t es = part_bytes(k);
  auto moves = [&](int t) { return part_ptr(L.tensors[t], k) != nullptr && !((resident[t] >> k) & 1); };
  int t = t0;
  while (t < t1) {
    char* h = static_cast<char*>(part_ptr(L.tensors[t], k));
    char* d = static_cast<char*>(part_ptr(slot[t], k));
    if (!moves(t)) {
      ++t;
      continue;
    }
    size_t bytes = es * (size_t)L.tensors[t].numel;
    int u = t + 1;
    while (u < t1 && moves(u) && part_ptr(L.tensors[u], k) == h + bytes && part_ptr(slot[u], k) == d + bytes) {
      bytes += es * (size_t)L.tensors[u].numel;
      ++u;
    }
    if (kind == cudaMemcpyHostToDevice) SF_TRY(copy_async(d, h, bytes, kind, s, what));
    else SF_TRY(copy_async(h, d, bytes, kind, s, what));
    t = u;
  }
  return SF_OK;
}

void destroy_events(sf_window_s* w) {
  for (auto* v : {&w->ev_in, &w->ev_done, &w->ev_free, &w->ev_layer})
    for (cudaEvent_t e : *v)
      if (e) cudaEventDestroy(e);
}

sf_status new_event(cudaEvent_t* e) {
  cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
  return r == cudaSuccess ? SF_OK : sf::cuda_fail(r, "cudaEventCreate");
}

sf_status check_layer(const sf_window_s* w, const sf_host_layer& L, int li, const uint8_t* resident) {
  if (L.n_tensors < 0 || L.n_tensors > w->n_tensors)
    return sf::fail(SF_ERR_INVALID, "layer %d: %d tensors, window slots hold %d", li, L.n_tensors,
                    w->n_tensors);
  if (L.n_tensors > 0 && !L.tensors) return sf::fail(SF_ERR_INVALID, "layer %d: tensors is NULL", li);
  for (int t = 0; t < L.n_tensors; ++t) {
    const sf_tensor& h = L.tensors[t];
    if (h.numel < 0) return sf::fail(SF_ERR_INVALID, "layer %d tensor %d: numel < 0", li, t);
    if (h.numel == 0) continue;
    if (!h.grad || !h.master || !h.exp_avg || !h.exp_avg_sq)
      return sf::fail(SF_ERR_INVALID, "layer %d tensor %d: NULL host array", li, t);
    for (const auto& slot : w->slots) {
      const sf_tensor& d = slot[t];
      if (h.numel > d.numel)
        return sf::fail(SF_ERR_INVALID, "layer %d tensor %d: numel %lld exceeds slot capacity %lld",
                        li, t, (long long)h.numel, (long long)d.numel);
      // a slot array may be NULL only where the layer's array is device-resident
      for (int k = kGrad; k <= kWeight; ++k)
        if (part_ptr(h, (Part)k) && !((resident[t] >> k) & 1) && !part_ptr(d, (Part)k))
          return sf::fail(SF_ERR_INVALID, "layer %d tensor %d: array %d is in host memory but the slot has no buffer "
                                          "for it", li, t, k);
    }
  }
  return SF_OK;
}

// Bit k of out[t]: array k of tensor t of the layer is in this device's memory.
void residency(const sf_host_layer& L, uint8_t* out) {
  for (int t = 0; t < L.n_tensors; ++t) {
    uint8_t r = 0;
    for (int k = kGrad; k <= kWeight; ++k) {
      const void* p = part_ptr(L.tensors[t], (Part)k);
      if (p && sf::on_current_device(p)) r |= (uint8_t)(1u << k);
    }
    out[t] = r;
  }
}

}  // namespace

extern "C" {

sf_status sf_window_create(int n_slots, const sf_tensor* const* device_slots, int n_tensors_per_slot,
                           void* h2d_stream, void* compute_stream, void* d2h_stream,
                           sf_window* out) {
  sf::clear_error();
  if (!out) return sf::fail(SF_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (n_slots < 1) return sf::fail(SF_ERR_INVALID, "n_slots must be >= 1");
  if (n_tensors_per_slot < 0) return sf::fail(SF_ERR_INVALID, "n_tensors_per_slot < 0");
  if (!device_slots) return sf::fail(SF_ERR_INVALID, "device_slots is NULL");
  sf_window_s* w = new (std::nothrow) sf_window_s;
  if (!w) return sf::fail(SF_ERR_OOM, "window allocation failed");
  cudaGetDevice(&w->device);
  w->n_slots = n_slots;
  w->n_tensors = n_tensors_per_slot;
  w->h2d = sf::as_stream(h2d_stream);
  w->comp = sf::as_stream(compute_stream);
  w->d2h = sf::as_stream(d2h_stream);
  for (int s = 0; s < n_slots; ++s) {
    if (n_tensors_per_slot > 0 && !device_slots[s]) {
      delete w;
      return sf::fail(SF_ERR_INVALID, "slot %d is NULL", s);
    }
    w->slots.emplace_back(device_slots[s], device_slots[s] + n_tensors_per_slot);
  }
  const int ne = n_slots * std::max(1, n_tensors_per_slot);
  w->ev_in.assign(ne, nullptr);
  w->ev_done.assign(ne, nullptr);
  w->ev_free.assign(ne, nullptr);
  w->free_gen.assign(ne, 0);
  for (int e = 0; e < ne; ++e) {
    sf_status st = SF_OK;
    if ((st = new_event(&w->ev_in[e])) != SF_OK || (st = new_event(&w->ev_done[e])) != SF_OK ||
        (st = new_event(&w->ev_free[e])) != SF_OK) {
      destroy_events(w);
      delete w;
      return st;
    }
  }
  *out = w;
  return SF_OK;
}

sf_status sf_slide_window_step(sf_window w, const sf_host_layer* layers, int n_layers,
                               const int32_t* order, int n_order, const sf_adamw_hparams* hp,
                               int64_t* steps) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("sf_slide_window_step");
  if (!w) return sf::fail(SF_ERR_INVALID, "window is NULL");
  if (n_order < 0 || n_layers < 0) return sf::fail(SF_ERR_INVALID, "negative count");
  if (n_order == 0) return SF_OK;
  if (!layers || !order || !steps) return sf::fail(SF_ERR_INVALID, "NULL array");
  sf::AdamConsts probe;
  SF_TRY(sf::make_adam_consts(hp, 1, true, &probe));  // validates hp before enqueueing
  for (int v = 0; v < n_order; ++v)
    if (order[v] < 0 || order[v] >= n_layers)
      return sf::fail(SF_ERR_INVALID, "order[%d] = %d out of [0, %d)", v, order[v], n_layers);
  // which arrays of each layer are already in this device's memory
  std::vector<uint8_t> resident((size_t)n_layers * std::max(1, w->n_tensors), 0);
  for (int l = 0; l < n_layers; ++l) {
    if (layers[l].n_tensors > 0 && layers[l].n_tensors <= w->n_tensors && layers[l].tensors)
      residency(layers[l], resident.data() + (size_t)l * w->n_tensors);
    SF_TRY(check_layer(w, layers[l], l, resident.data() + (size_t)l * w->n_tensors));
    if (steps[l] < 0) return sf::fail(SF_ERR_INVALID, "steps[%d] < 0", l);
  }
  if ((int)w->ev_layer.size() < n_layers) {
    int old = (int)w->ev_layer.size();
    w->ev_layer.resize(n_layers, nullptr);
    w->layer_pending.resize(n_layers, false);
    for (int l = old; l < n_layers; ++l) SF_TRY(new_event(&w->ev_layer[l]));
  }

  std::vector<sf_tensor> dev(w->n_tensors);
  for (int v = 0; v < n_order; ++v) {
    const int l = order[v];
    const int s = (int)(w->visits % w->n_slots);
    const sf_host_layer& L = layers[l];
    const std::vector<sf_tensor>& slot = w->slots[s];
    const int eb = s * w->n_tensors;          // this slot's events
    const int64_t step = steps[l] + 1;
    // arrays already in this device's memory are used in place
    const uint8_t* res = resident.data() + (size_t)l * w->n_tensors;

    // the previous write-back of this layer must have landed before it is read again
    if (w->layer_pending[l])
      SF_CUDA_TRY(cudaStreamWaitEvent(w->h2d, w->ev_layer[l], 0), "wait layer write-back");
    int t0 = 0;
    while (t0 < L.n_tensors) {
      int t1 = t0;
      int64_t params = 0;
      while (t1 < L.n_tensors && (params < kGroupParams || t1 == t0)) params += L.tensors[t1++].numel;

      // h2d: the slot's tensors of this group are free (one wait per distinct
      // earlier group that held them), then copy in
      int64_t last = -1;
      for (int t = t0; t < t1; ++t) {
        const int64_t g = w->free_gen[eb + t];
        if (g > 0 && g != last)
          SF_CUDA_TRY(cudaStreamWaitEvent(w->h2d, w->ev_free[eb + t], 0), "wait slot tensor free");
        last = g;
      }
      SF_TRY(copy_runs(L, slot, res, t0, t1, kGrad, cudaMemcpyHostToDevice, w->h2d, "h2d grad"));
      SF_TRY(copy_runs(L, slot, res, t0, t1, kMaster, cudaMemcpyHostToDevice, w->h2d, "h2d master"));
      SF_TRY(copy_runs(L, slot, res, t0, t1, kExpAvg, cudaMemcpyHostToDevice, w->h2d, "h2d exp_avg"));
      SF_TRY(copy_runs(L, slot, res, t0, t1, kExpAvgSq, cudaMemcpyHostToDevice, w->h2d, "h2d exp_avg_sq"));
      SF_CUDA_TRY(cudaEventRecord(w->ev_in[eb + t0], w->h2d), "record ev_in");

      // compute: the fused update of the group, on the slot's copy of each
      // array or on the array itself where it is device-resident
      SF_CUDA_TRY(cudaStreamWaitEvent(w->comp, w->ev_in[eb + t0], 0), "wait ev_in");
      for (int t = t0; t < t1; ++t) {
        const sf_tensor& h = L.tensors[t];
        const uint8_t r = res[t];
        dev[t] = slot[t];
        dev[t].numel = h.numel;
        if (r & (1u << kGrad)) dev[t].grad = h.grad;
        if (r & (1u << kMaster)) dev[t].master = h.master;
        if (r & (1u << kExpAvg)) dev[t].exp_avg = h.exp_avg;
        if (r & (1u << kExpAvgSq)) dev[t].exp_avg_sq = h.exp_avg_sq;
        if (!h.weight) dev[t].weight = nullptr;
        else if (r & (1u << kWeight)) dev[t].weight = h.weight;
      }
      SF_TRY(sf::adamw_layer_step_impl(dev.data() + t0, t1 - t0, hp, step, w->comp));
      SF_CUDA_TRY(cudaEventRecord(w->ev_done[eb + t0], w->comp), "record ev_done");

      // d2h: write the group back; each tensor of the slot is free when its copies end
      SF_CUDA_TRY(cudaStreamWaitEvent(w->d2h, w->ev_done[eb + t0], 0), "wait ev_done");
      SF_TRY(copy_runs(L, slot, res, t0, t1, kMaster, cudaMemcpyDeviceToHost, w->d2h, "d2h master"));
      SF_TRY(copy_runs(L, slot, res, t0, t1, kExpAvg, cudaMemcpyDeviceToHost, w->d2h, "d2h exp_avg"));
      SF_TRY(copy_runs(L, slot, res, t0, t1, kExpAvgSq, cudaMemcpyDeviceToHost, w->d2h, "d2h exp_avg_sq"));
      SF_TRY(copy_runs(L, slot, res, t0, t1, kWeight, cudaMemcpyDeviceToHost, w->d2h, "d2h weight"));
      const int64_t g = ++w->gen;
      for (int t = t0; t < t1; ++t) {
        SF_CUDA_TRY(cudaEventRecord(w->ev_free[eb + t], w->d2h), "record ev_free");
        w->free_gen[eb + t] = g;
      }
      t0 = t1;
    }
    steps[l] = step;
    SF_CUDA_TRY(cudaEventRecord(w->ev_layer[l], w->d2h), "record ev_layer");
    w->layer_pending[l] = true;
    ++w->visits;
  }
  return SF_OK;
}

sf_status sf_window_sync(sf_window w, int64_t timeout_ms) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("sf_window_sync");
  if (!w) return sf::fail(SF_ERR_INVALID, "window is NULL");
  SF_TRY(sf::bounded_wait_stream(w->h2d, timeout_ms, "window h2d stream"));
  SF_TRY(sf::bounded_wait_stream(w->comp, timeout_ms, "window compute stream"));
  SF_TRY(sf::bounded_wait_stream(w->d2h, timeout_ms, "window d2h stream"));
  return SF_OK;
}

sf_status sf_window_destroy(sf_window w) {
  sf::clear_error();
  if (!w) return SF_OK;
  sf_status st = sf_window_sync(w, 0);
  destroy_events(w);
  delete w;
  return st;
}

// Test hook: make the n-th copy the window enqueues from now on fail once
// (n >= 1), or switch the hook off (n = 0).  Host-side only: the failing
// copy is never handed to CUDA.
void sf_test_fail_copy_after(int64_t n) {
  g_copy_count = 0;
  g_fail_copy_at = n > 0 ? n : 0;
}

}  // extern "C"

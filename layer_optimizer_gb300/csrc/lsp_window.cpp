// Layer-wise schedule of the sparse-projector step with the compressed
// optimizer state in pinned host memory.
//
// LSP-Offload ("Practical offloading for fine-tuning LLM on commodity GPU
// via learned sparse projectors", abstract and method section) keeps only
// compressed quantities on the host, computes the update there in the
// compressed space, and schedules the transfers layer by layer so that
// communication overlaps the compute of neighbouring layers.  Every layer's
// compressed moments m~, v~ (d x d fp32) live in pinned host memory.  Two
// placements of the compressed AdamW:
//
//  * host update (lsp_window_create_host_update; the pages' own): the
//    compute stream compresses the layer's gradient into its slot, the d2h
//    stream brings S to the host, a host function ordered after that copy
//    runs the compressed AdamW on the host cores (a small persistent thread
//    pool) on m~, v~ in place, the h2d stream takes dS back, and the
//    compute stream decompress-applies it.  The compress of the next
//    n_slots - 1 layers is enqueued before this layer's decompress, so the
//    host round trip of one layer overlaps the next layers' GPU work.  Per
//    layer the link carries d*d*4 bytes each way and no moments.
//  * device update (lsp_window_create): m~, v~ come into the slot, the
//    compressed AdamW runs on the GPU, and they go back (2*d*d*4 bytes each
//    way per layer).
//
// The engine's only arithmetic is the host compressed step (host_adamw.cpp,
// bitwise the device kernel's); it calls lsp_compress and
// lsp_decompress_apply for the rest, allocates no device memory, and orders
// everything with CUDA events and stream-ordered host functions.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <functional>
#include <memory>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "common.h"

namespace {

// Fixed pool of host threads for the compressed update: run(total, f) splits
// [0, total) into one contiguous part per thread, the caller doing part 0,
// and returns when every part is done.
class HostPool {
 public:
  explicit HostPool(int n) : n_(n < 1 ? 1 : n) {}
  bool start() {
    try {
      for (int k = 1; k < n_; ++k) th_.emplace_back([this, k] { loop(k); });
    } catch (...) {
      stop();
      return false;
    }
    return true;
  }
  ~HostPool() { stop(); }
  void run(int64_t total, const std::function<void(int64_t, int64_t)>& f) {
    {
      std::unique_lock<std::mutex> lk(mu_);
      job_ = &f;
      total_ = total;
      remaining_ = n_ - 1;
      ++gen_;
    }
    cv_.notify_all();
    f(0, total / n_);
    std::unique_lock<std::mutex> lk(mu_);
    done_.wait(lk, [this] { return remaining_ == 0; });
    job_ = nullptr;
  }

 private:
  void loop(int k) {
    uint64_t seen = 0;
    for (;;) {
      const std::function<void(int64_t, int64_t)>* f;
      int64_t total;
      {
        std::unique_lock<std::mutex> lk(mu_);
        cv_.wait(lk, [&] { return quit_ || gen_ != seen; });
        if (quit_) return;
        seen = gen_;
        f = job_;
        total = total_;
      }
      (*f)(total * k / n_, total * (k + 1) / n_);
      std::lock_guard<std::mutex> lk(mu_);
      if (--remaining_ == 0) done_.notify_one();
    }
  }
  void stop() {
    {
      std::lock_guard<std::mutex> lk(mu_);
      quit_ = true;
    }
    cv_.notify_all();
    for (auto& t : th_)
      if (t.joinable()) t.join();
    th_.clear();
  }
  int n_;
  std::vector<std::thread> th_;
  std::mutex mu_;
  std::condition_variable cv_, done_;
  const std::function<void(int64_t, int64_t)>* job_ = nullptr;
  int64_t total_ = 0;
  int remaining_ = 0;
  uint64_t gen_ = 0;
  bool quit_ = false;
};

// Timeline points per visit: compress start/end, S copy start/end, host
// update end, dS copy start/end, decompress-apply start/end.
constexpr int kTimelinePoints = 9;

// One host update: read by a host function when the stream reaches it.
struct HostJob {
  HostPool* pool = nullptr;
  const float* S = nullptr;
  float* m = nullptr;
  float* v = nullptr;
  float* dS = nullptr;
  int64_t n = 0;
  sf::AdamConsts c{};
  std::atomic<int64_t>* done = nullptr;
};

// Jobs in flight at most (a ring; the host waits, bounded, if the GPU side
// falls this far behind).
constexpr int64_t kJobRing = 1024;

}  // namespace

struct lsp_window_s {
  int n_slots = 0;
  int32_t d = 0;
  bool host_update = false;
  std::vector<lsp_slot> slots;
  std::vector<lsp_host_slot> hslots;
  std::unique_ptr<HostPool> pool;
  std::vector<HostJob> jobs;
  std::atomic<int64_t> jobs_done{0};
  int64_t jobs_issued = 0;
  // host-update mode, per slot: S ready / S copied out / dS ready on the
  // host / dS copied in / decompress-apply done
  std::vector<cudaEvent_t> ev_S, ev_S_out, ev_dS_host, ev_dS_in, ev_apply;
  // optional timeline (measurement): kTimelinePoints timing events per visit
  std::vector<cudaEvent_t> tl_ev;
  int tl_capacity = 0, tl_used = 0;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  std::vector<cudaEvent_t> ev_in, ev_moments, ev_free;   // per slot
  std::vector<bool> slot_used;
  std::vector<cudaEvent_t> ev_layer;                      // a layer's moments are back on the host
  std::vector<bool> layer_pending;
  int64_t visits = 0;
};

namespace {

sf_status new_event(cudaEvent_t* e) {
  cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
  return r == cudaSuccess ? SF_OK : sf::cuda_fail(r, "cudaEventCreate");
}

void destroy_events(lsp_window_s* w) {
  for (auto* v : {&w->ev_in, &w->ev_moments, &w->ev_free, &w->ev_layer, &w->ev_S, &w->ev_S_out, &w->ev_dS_host,
                  &w->ev_dS_in, &w->ev_apply, &w->tl_ev})
    for (cudaEvent_t e : *v)
      if (e) cudaEventDestroy(e);
}

// Host function: the compressed AdamW of one layer on the host cores.
void CUDART_CB run_host_update(void* p) {
  HostJob* j = static_cast<HostJob*>(p);
  const HostJob job = *j;
  job.pool->run(job.n, [&](int64_t b, int64_t e) { sf::host_adamw_compressed(job.S, job.m, job.v, job.dS, b, e, job.c); });
  job.done->fetch_add(1, std::memory_order_release);
}

sf_status check_layer(const lsp_window_s* w, const lsp_layer& L, int li) {
  if (!L.P || !L.Q || !L.G || !L.W || !L.m_host || !L.v_host)
    return sf::fail(SF_ERR_INVALID, "lsp layer %d: NULL projector or array", li);
  if (lsp_projector_dim(L.P) != w->d || lsp_projector_dim(L.Q) != w->d)
    return sf::fail(SF_ERR_INVALID, "lsp layer %d: projector d differs from the window's d = %d", li, w->d);
  if (lsp_projector_rows(L.P) != L.m || lsp_projector_rows(L.Q) != L.n)
    return sf::fail(SF_ERR_INVALID, "lsp layer %d: projector rows do not match m, n", li);
  const size_t need = lsp_workspace_bytes(L.m, L.n, w->d);
  for (const lsp_slot& s : w->slots)
    if (s.ws_bytes < need)
      return sf::fail(SF_ERR_INVALID, "lsp layer %d needs %zu workspace bytes, a slot has %zu", li, need,
                      s.ws_bytes);
  for (const lsp_host_slot& s : w->hslots)
    if (s.ws_bytes < need)
      return sf::fail(SF_ERR_INVALID, "lsp layer %d needs %zu workspace bytes, a slot has %zu", li, need,
                      s.ws_bytes);
  return SF_OK;
}

// The host-update schedule (see the file comment).  Visit u's front half
// (compress, S out, host update, dS in) is enqueued before the back half
// (decompress-apply) of visit u - (n_slots - 1).
// Records timeline point `k` of timeline visit `tv` on stream `st` (if the
// timeline is on and has room).  A point is recorded before the event another
// stream waits on, so points of one visit come out in causal order.
sf_status mark(lsp_window_s* w, int tv, int k, cudaStream_t st) {
  if (tv < 0 || tv >= w->tl_capacity) return SF_OK;
  SF_CUDA_TRY(cudaEventRecord(w->tl_ev[(size_t)tv * kTimelinePoints + k], st), "record timeline event");
  return SF_OK;
}

sf_status enqueue_front(lsp_window_s* w, const lsp_layer& L, int s, const sf_adamw_hparams* hp, int64_t step,
                        bool reused, int tv) {
  const lsp_host_slot& slot = w->hslots[s];
  const size_t dd = (size_t)w->d * w->d * sizeof(float);
  // compute: the slot's S has been copied out by its previous visit
  if (reused) SF_CUDA_TRY(cudaStreamWaitEvent(w->comp, w->ev_S_out[s], 0), "wait S out");
  SF_TRY(mark(w, tv, 0, w->comp));
  SF_TRY(lsp_compress(L.P, L.Q, L.G, L.g_dtype, L.m, L.n, slot.S, slot.ws, slot.ws_bytes, w->comp));
  SF_TRY(mark(w, tv, 1, w->comp));
  SF_CUDA_TRY(cudaEventRecord(w->ev_S[s], w->comp), "record ev_S");
  // d2h: S to the host, once the previous visit's dS has left the staging buffer
  SF_CUDA_TRY(cudaStreamWaitEvent(w->d2h, w->ev_S[s], 0), "wait ev_S");
  if (reused) SF_CUDA_TRY(cudaStreamWaitEvent(w->d2h, w->ev_dS_in[s], 0), "wait dS in");
  SF_TRY(mark(w, tv, 2, w->d2h));
  SF_CUDA_TRY(cudaMemcpyAsync(slot.S_host, slot.S, dd, cudaMemcpyDeviceToHost, w->d2h), "d2h S");
  SF_TRY(mark(w, tv, 3, w->d2h));
  SF_CUDA_TRY(cudaEventRecord(w->ev_S_out[s], w->d2h), "record ev_S_out");
  // host: the compressed AdamW on the layer's moments, ordered after the copy
  if (w->jobs_issued >= kJobRing) {
    const int64_t need = w->jobs_issued - kJobRing + 1;
    const auto t0 = std::chrono::steady_clock::now();
    while (w->jobs_done.load(std::memory_order_acquire) < need) {
      if (std::chrono::duration_cast<std::chrono::milliseconds>(std::chrono::steady_clock::now() - t0).count() >
          sf::default_timeout_ms())
        return sf::fail(SF_ERR_TIMEOUT, "host updates are %lld behind", (long long)kJobRing);
      std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
  }
  HostJob& job = w->jobs[w->jobs_issued % kJobRing];
  job.pool = w->pool.get();
  job.S = slot.S_host;
  job.m = L.m_host;
  job.v = L.v_host;
  job.dS = slot.dS_host;
  job.n = (int64_t)w->d * w->d;
  SF_TRY(sf::make_adam_consts(hp, step, false, &job.c));
  job.done = &w->jobs_done;
  SF_CUDA_TRY(cudaLaunchHostFunc(w->d2h, run_host_update, &job), "cudaLaunchHostFunc (host update)");
  ++w->jobs_issued;
  SF_TRY(mark(w, tv, 4, w->d2h));
  SF_CUDA_TRY(cudaEventRecord(w->ev_dS_host[s], w->d2h), "record ev_dS_host");
  // h2d: dS back into the slot, once the previous visit's apply has read it
  SF_CUDA_TRY(cudaStreamWaitEvent(w->h2d, w->ev_dS_host[s], 0), "wait ev_dS_host");
  if (reused) SF_CUDA_TRY(cudaStreamWaitEvent(w->h2d, w->ev_apply[s], 0), "wait apply");
  SF_TRY(mark(w, tv, 5, w->h2d));
  SF_CUDA_TRY(cudaMemcpyAsync(slot.dS, slot.dS_host, dd, cudaMemcpyHostToDevice, w->h2d), "h2d dS");
  SF_TRY(mark(w, tv, 6, w->h2d));
  SF_CUDA_TRY(cudaEventRecord(w->ev_dS_in[s], w->h2d), "record ev_dS_in");
  return SF_OK;
}

sf_status enqueue_back(lsp_window_s* w, const lsp_layer& L, int s, int tv) {
  const lsp_host_slot& slot = w->hslots[s];
  SF_CUDA_TRY(cudaStreamWaitEvent(w->comp, w->ev_dS_in[s], 0), "wait ev_dS_in");
  SF_TRY(mark(w, tv, 7, w->comp));
  SF_TRY(lsp_decompress_apply(L.P, L.Q, slot.dS, L.W, L.w_dtype, L.w_bf16_mirror, L.m, L.n, slot.ws, slot.ws_bytes,
                              w->comp));
  SF_TRY(mark(w, tv, 8, w->comp));
  SF_CUDA_TRY(cudaEventRecord(w->ev_apply[s], w->comp), "record ev_apply");
  return SF_OK;
}

}  // namespace

extern "C" {

sf_status lsp_window_create(int n_slots, const lsp_slot* slots, int32_t d, void* h2d_stream,
                            void* compute_stream, void* d2h_stream, lsp_window* out) {
  sf::clear_error();
  if (!out) return sf::fail(SF_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (n_slots < 1 || !slots) return sf::fail(SF_ERR_INVALID, "need n_slots >= 1 and a slot array");
  if (d < 1) return sf::fail(SF_ERR_INVALID, "d must be >= 1");
  for (int s = 0; s < n_slots; ++s)
    if (!slots[s].S || !slots[s].m || !slots[s].v || !slots[s].dS || !slots[s].ws)
      return sf::fail(SF_ERR_INVALID, "slot %d has a NULL buffer", s);
  lsp_window_s* w = new (std::nothrow) lsp_window_s;
  if (!w) return sf::fail(SF_ERR_OOM, "window allocation failed");
  w->n_slots = n_slots;
  w->d = d;
  w->slots.assign(slots, slots + n_slots);
  w->h2d = sf::as_stream(h2d_stream);
  w->comp = sf::as_stream(compute_stream);
  w->d2h = sf::as_stream(d2h_stream);
  w->ev_in.assign(n_slots, nullptr);
  w->ev_moments.assign(n_slots, nullptr);
  w->ev_free.assign(n_slots, nullptr);
  w->slot_used.assign(n_slots, false);
  for (int s = 0; s < n_slots; ++s) {
    sf_status st = SF_OK;
    if ((st = new_event(&w->ev_in[s])) != SF_OK || (st = new_event(&w->ev_moments[s])) != SF_OK ||
        (st = new_event(&w->ev_free[s])) != SF_OK) {
      destroy_events(w);
      delete w;
      return st;
    }
  }
  *out = w;
  return SF_OK;
}

sf_status lsp_window_create_host_update(int n_slots, const lsp_host_slot* slots, int32_t d, int n_threads,
                                        void* h2d_stream, void* compute_stream, void* d2h_stream, lsp_window* out) {
  sf::clear_error();
  if (!out) return sf::fail(SF_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (n_slots < 1 || !slots) return sf::fail(SF_ERR_INVALID, "need n_slots >= 1 and a slot array");
  if (d < 1) return sf::fail(SF_ERR_INVALID, "d must be >= 1");
  for (int s = 0; s < n_slots; ++s)
    if (!slots[s].S || !slots[s].dS || !slots[s].S_host || !slots[s].dS_host || !slots[s].ws)
      return sf::fail(SF_ERR_INVALID, "slot %d has a NULL buffer", s);
  lsp_window_s* w = new (std::nothrow) lsp_window_s;
  if (!w) return sf::fail(SF_ERR_OOM, "window allocation failed");
  w->n_slots = n_slots;
  w->d = d;
  w->host_update = true;
  w->hslots.assign(slots, slots + n_slots);
  w->h2d = sf::as_stream(h2d_stream);
  w->comp = sf::as_stream(compute_stream);
  w->d2h = sf::as_stream(d2h_stream);
  w->slot_used.assign(n_slots, false);
  w->jobs.resize(kJobRing);
  w->pool.reset(new (std::nothrow) HostPool(n_threads > 0 ? n_threads : std::min(8, sf::usable_cores())));
  if (!w->pool || !w->pool->start()) {
    delete w;
    return sf::fail(SF_ERR_OOM, "could not start the host update threads");
  }
  for (auto* v : {&w->ev_S, &w->ev_S_out, &w->ev_dS_host, &w->ev_dS_in, &w->ev_apply}) v->assign(n_slots, nullptr);
  for (int s = 0; s < n_slots; ++s)
    for (auto* v : {&w->ev_S, &w->ev_S_out, &w->ev_dS_host, &w->ev_dS_in, &w->ev_apply}) {
      sf_status st = new_event(&(*v)[s]);
      if (st != SF_OK) {
        destroy_events(w);
        delete w;
        return st;
      }
    }
  *out = w;
  return SF_OK;
}

sf_status lsp_slide_window_step(lsp_window w, const lsp_layer* layers, int n_layers, const int32_t* order,
                                int n_order, const sf_adamw_hparams* hp, int64_t* steps) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("lsp_slide_window_step");
  if (!w) return sf::fail(SF_ERR_INVALID, "window is NULL");
  if (n_order < 0 || n_layers < 0) return sf::fail(SF_ERR_INVALID, "negative count");
  if (n_order == 0) return SF_OK;
  if (!layers || !order || !steps) return sf::fail(SF_ERR_INVALID, "NULL array");
  sf::AdamConsts probe;
  SF_TRY(sf::make_adam_consts(hp, 1, false, &probe));
  for (int v = 0; v < n_order; ++v)
    if (order[v] < 0 || order[v] >= n_layers)
      return sf::fail(SF_ERR_INVALID, "order[%d] = %d out of [0, %d)", v, order[v], n_layers);
  for (int l = 0; l < n_layers; ++l) {
    SF_TRY(check_layer(w, layers[l], l));
    if (steps[l] < 0) return sf::fail(SF_ERR_INVALID, "steps[%d] < 0", l);
  }
  if ((int)w->ev_layer.size() < n_layers) {
    const int old = (int)w->ev_layer.size();
    w->ev_layer.resize(n_layers, nullptr);
    w->layer_pending.resize(n_layers, false);
    for (int l = old; l < n_layers; ++l) SF_TRY(new_event(&w->ev_layer[l]));
  }
  if (w->host_update) {
    // visit u's front half, then the back half of visit u - (n_slots - 1)
    const int look = w->n_slots - 1;
    std::vector<int> slot_of(n_order);
    const int tv0 = w->tl_used;                 // timeline index of this call's first visit
    for (int u = 0; u < n_order + look; ++u) {
      if (u < n_order) {
        const int l = order[u];
        const int s = (int)(w->visits % w->n_slots);
        slot_of[u] = s;
        const int64_t step = steps[l] + 1;
        SF_TRY(enqueue_front(w, layers[l], s, hp, step, w->slot_used[s], tv0 + u));
        w->slot_used[s] = true;
        steps[l] = step;
        ++w->visits;
      }
      const int b = u - look;
      if (b >= 0) SF_TRY(enqueue_back(w, layers[order[b]], slot_of[b], tv0 + b));
    }
    if (w->tl_capacity > 0) w->tl_used = std::min(w->tl_capacity, tv0 + n_order);
    return SF_OK;
  }
  const size_t dd = (size_t)w->d * w->d * sizeof(float);
  for (int v = 0; v < n_order; ++v) {
    const int l = order[v];
    const int s = (int)(w->visits % w->n_slots);
    const lsp_layer& L = layers[l];
    const lsp_slot& slot = w->slots[s];
    const int64_t step = steps[l] + 1;

    // compute: compress the layer's gradient into the slot
    SF_TRY(lsp_compress(L.P, L.Q, L.G, L.g_dtype, L.m, L.n, slot.S, slot.ws, slot.ws_bytes, w->comp));

    // h2d: the slot's moments are free and the layer's last write-back landed
    if (w->slot_used[s]) SF_CUDA_TRY(cudaStreamWaitEvent(w->h2d, w->ev_free[s], 0), "wait slot free");
    if (w->layer_pending[l])
      SF_CUDA_TRY(cudaStreamWaitEvent(w->h2d, w->ev_layer[l], 0), "wait layer write-back");
    SF_CUDA_TRY(cudaMemcpyAsync(slot.m, L.m_host, dd, cudaMemcpyHostToDevice, w->h2d), "h2d m");
    SF_CUDA_TRY(cudaMemcpyAsync(slot.v, L.v_host, dd, cudaMemcpyHostToDevice, w->h2d), "h2d v");
    SF_CUDA_TRY(cudaEventRecord(w->ev_in[s], w->h2d), "record ev_in");

    // compute: the compressed step, then decompress-apply
    SF_CUDA_TRY(cudaStreamWaitEvent(w->comp, w->ev_in[s], 0), "wait ev_in");
    SF_TRY(lsp_adamw_compressed(slot.S, slot.m, slot.v, slot.dS, (int64_t)w->d * w->d, hp, step, w->comp));
    SF_CUDA_TRY(cudaEventRecord(w->ev_moments[s], w->comp), "record ev_moments");
    SF_TRY(lsp_decompress_apply(L.P, L.Q, slot.dS, L.W, L.w_dtype, L.w_bf16_mirror, L.m, L.n, slot.ws,
                                slot.ws_bytes, w->comp));

    // d2h: the moments go back as soon as the compressed step wrote them
    SF_CUDA_TRY(cudaStreamWaitEvent(w->d2h, w->ev_moments[s], 0), "wait ev_moments");
    SF_CUDA_TRY(cudaMemcpyAsync(L.m_host, slot.m, dd, cudaMemcpyDeviceToHost, w->d2h), "d2h m");
    SF_CUDA_TRY(cudaMemcpyAsync(L.v_host, slot.v, dd, cudaMemcpyDeviceToHost, w->d2h), "d2h v");
    SF_CUDA_TRY(cudaEventRecord(w->ev_free[s], w->d2h), "record ev_free");
    SF_CUDA_TRY(cudaEventRecord(w->ev_layer[l], w->d2h), "record ev_layer");
    w->slot_used[s] = true;
    w->layer_pending[l] = true;
    steps[l] = step;
    ++w->visits;
  }
  return SF_OK;
}

sf_status lsp_window_timeline_start(lsp_window w, int capacity) {
  sf::clear_error();
  if (!w) return sf::fail(SF_ERR_INVALID, "window is NULL");
  if (!w->host_update) return sf::fail(SF_ERR_INVALID, "the timeline is kept by host-update windows only");
  if (capacity < 0 || capacity > (1 << 20)) return sf::fail(SF_ERR_INVALID, "capacity must be in [0, 2^20]");
  SF_TRY(lsp_window_sync(w, 0));
  for (cudaEvent_t e : w->tl_ev)
    if (e) cudaEventDestroy(e);
  w->tl_ev.assign((size_t)capacity * kTimelinePoints, nullptr);
  w->tl_capacity = 0;
  w->tl_used = 0;
  for (cudaEvent_t& e : w->tl_ev) SF_CUDA_TRY(cudaEventCreate(&e), "cudaEventCreate (timeline)");
  w->tl_capacity = capacity;
  return SF_OK;
}

sf_status lsp_window_timeline_read(lsp_window w, float* ms, int capacity, int* n_visits) {
  sf::clear_error();
  if (!w || !n_visits || (!ms && capacity > 0)) return sf::fail(SF_ERR_INVALID, "NULL argument");
  *n_visits = 0;
  if (w->tl_used == 0) return SF_OK;
  SF_TRY(lsp_window_sync(w, 0));
  const int n = std::min(capacity, w->tl_used);
  cudaEvent_t base = w->tl_ev[0];
  for (int v = 0; v < n; ++v)
    for (int k = 0; k < kTimelinePoints; ++k) {
      float t = 0.0f;
      SF_CUDA_TRY(cudaEventElapsedTime(&t, base, w->tl_ev[(size_t)v * kTimelinePoints + k]), "timeline elapsed time");
      ms[(size_t)v * kTimelinePoints + k] = t;
    }
  *n_visits = n;
  return SF_OK;
}

sf_status lsp_window_sync(lsp_window w, int64_t timeout_ms) {
  sf::clear_error();
  sf::NvtxRange nvtx_range("lsp_window_sync");
  if (!w) return sf::fail(SF_ERR_INVALID, "window is NULL");
  SF_TRY(sf::bounded_wait_stream(w->h2d, timeout_ms, "lsp window h2d stream"));
  SF_TRY(sf::bounded_wait_stream(w->comp, timeout_ms, "lsp window compute stream"));
  SF_TRY(sf::bounded_wait_stream(w->d2h, timeout_ms, "lsp window d2h stream"));
  return SF_OK;
}

sf_status lsp_window_destroy(lsp_window w) {
  sf::clear_error();
  if (!w) return SF_OK;
  sf_status st = lsp_window_sync(w, 0);
  // work still in flight may yet run host updates that read the window:
  // keep it (the caller may destroy it again later)
  if (st == SF_ERR_TIMEOUT) return st;
  destroy_events(w);
  delete w;
  return st;
}

}  // extern "C"

// Layer-wise schedule of the sparse-projector step with the compressed
// optimizer state in pinned host memory.
//
// LSP-Offload ("Practical offloading for fine-tuning LLM on commodity GPU
// via learned sparse projectors", abstract and method section) keeps only
// compressed quantities on the host and schedules their transfers layer by
// layer so that communication overlaps the compute of neighbouring layers.
// Here every layer's compressed moments m~, v~ (d x d fp32) live in pinned
// host memory and pass through a small set of device slots: the compute
// stream compresses the layer's gradient into its slot while the h2d stream
// brings the layer's moments in; the compressed AdamW and the
// decompress-apply follow on the compute stream, and the d2h stream writes
// the moments back as soon as the compressed step has produced them.  The
// engine does no arithmetic of its own (it calls lsp_compress,
// lsp_adamw_compressed and lsp_decompress_apply), allocates nothing per
// call, and orders everything with CUDA events only.
#include <new>
#include <vector>

#include "common.h"

struct lsp_window_s {
  int n_slots = 0;
  int32_t d = 0;
  std::vector<lsp_slot> slots;
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
  for (auto* v : {&w->ev_in, &w->ev_moments, &w->ev_free, &w->ev_layer})
    for (cudaEvent_t e : *v)
      if (e) cudaEventDestroy(e);
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
  destroy_events(w);
  delete w;
  return st;
}

}  // extern "C"

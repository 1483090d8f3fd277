/*
 * sfopt.h -- C ABI of the GB300 (sm_103a) per-layer gradient-to-update step.
 *
 * Two modes of the same step, plus the engine that slides layers through
 * device memory:
 *
 *  (a) fused AdamW: bf16 gradient -> fp32 master weights and Adam moments
 *      -> bf16 weights, for all tensors of one layer in one launch.
 *      Follows "An Efficient Heterogeneous Co-Design for Fine-Tuning on a
 *      Single GPU" (SlideFormer), technical summary section 2.A (the layer
 *      update that the sliding engine overlaps with the next layer's
 *      compute) and 2.B (flattened fp32 optimizer states; fp32 -> bf16 type
 *      conversion).  The update is Adam with bias correction (Kingma & Ba
 *      2015, Algorithm 1) and decoupled weight decay (Loshchilov & Hutter
 *      2019, Algorithm 2).
 *
 *  (b) learned sparse projectors: S = P^T G Q, AdamW on S in the d x d
 *      compressed space, W -= P dS Q^T.  Follows "Practical offloading for
 *      fine-tuning LLM on commodity GPU via learned sparse projectors"
 *      (LSP-Offload), abstract and method section ("sparse projectors",
 *      "compress, compute in compressed space, decompress").
 *
 *  (c) the layer-sliding window: layers live in pinned host memory and are
 *      streamed through a fixed set of pre-allocated device slots on side
 *      streams while the update kernels run (SlideFormer, section 2.A
 *      "sliding window", "overlap of compute, transfer and update";
 *      section 2.B "pre-allocated GPU cache queue").
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Ownership: the caller owns every tensor buffer (device memory and
 *    pinned host memory) and every stream.  The library owns only the
 *    opaque handles it returns (projector index structures, window
 *    events), released by the matching *_destroy call.
 *  - Streams are passed as `void*` holding a cudaStream_t (NULL = the
 *    legacy default stream).  Every compute call is stream-ordered and
 *    asynchronous: it returns once its kernels are enqueued.
 *  - Errors: every call returns an sf_status.  Argument errors are found on
 *    the host before anything is enqueued (nothing is modified).  Launch
 *    errors return SF_ERR_CUDA; errors raised while kernels run surface at
 *    the next call that checks, or at sf_sync_status().  sf_last_error()
 *    gives a message for the calling thread's last failure.  No C++
 *    exception crosses this boundary.
 *  - Layouts are dense and row-major; element counts are int64.
 *  - Floating-point results are deterministic: the same inputs give the
 *    same bits on every run (no atomics in any reduction).
 */
#ifndef SFOPT_H
#define SFOPT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SF_OK = 0,
  SF_ERR_INVALID = -1,     /* null pointer, bad size, step < 1, bad index... */
  SF_ERR_CUDA = -2,        /* a CUDA launch or runtime error                 */
  SF_ERR_OOM = -3,         /* the library could not allocate its handle      */
  SF_ERR_UNSUPPORTED = -4, /* a size or dtype outside what a kernel supports */
  SF_ERR_TIMEOUT = -5      /* a bounded host wait ran out                    */
} sf_status;

typedef enum { SF_BF16 = 0, SF_FP32 = 1 } sf_dtype;

/* AdamW hyper-parameters.  Given in double; the library derives the fp32
 * constants the kernels use (1-beta1, 1-beta2, 1-lr*wd, lr/(1-beta1^t),
 * 1/sqrt(1-beta2^t)) in double and rounds each once. */
typedef struct {
  double lr;
  double beta1;
  double beta2;
  double eps;
  double weight_decay;
} sf_adamw_hparams;

/* One parameter tensor of a layer, flattened to `numel` elements.
 *   grad       : bf16 [numel], read
 *   master     : fp32 [numel], read + written (master weights theta)
 *   exp_avg    : fp32 [numel], read + written (first moment m)
 *   exp_avg_sq : fp32 [numel], read + written (second moment v)
 *   weight     : bf16 [numel], written (RNE of the new master); may be NULL
 * Pointers are device pointers for sf_adamw_layer_step and the device slots
 * of a window, pinned host pointers for the host layers of a window.  The
 * arrays must not overlap.  Any alignment is accepted; 16-byte aligned
 * arrays take the 128-bit path. */
typedef struct {
  const void* grad;
  float* master;
  float* exp_avg;
  float* exp_avg_sq;
  void* weight;
  int64_t numel;
} sf_tensor;

/* ------------------------------------------------------------------------
 * (a) Fused multi-tensor AdamW over one layer.
 *
 * Applies, per element, with t = `step` (>= 1):
 *   theta <- theta * (1 - lr*wd)
 *   m     <- beta1*m + (1-beta1)*g
 *   v     <- beta2*v + (1-beta2)*g^2
 *   theta <- theta - (lr/(1-beta1^t)) * m / (sqrt(v)/sqrt(1-beta2^t) + eps)
 *   weight = RNE_bf16(theta)
 * over all `n_tensors` tensors of the layer, in one kernel launch per
 * SF_MAX_TENSORS_PER_LAUNCH tensors.  Empty tensors (numel 0) are allowed.
 * Returns SF_ERR_INVALID for n_tensors < 0, a NULL array, a negative numel,
 * step < 1, or non-finite hyper-parameters.
 * The arrays may also be in pinned host memory (cudaHostAlloc / registered):
 * they are then updated in place over the host link by zero-copy loads and
 * stores (same arithmetic and bits; on GB300 about half the rate of the
 * copy-engine window, sf_slide_window_step).
 * ---------------------------------------------------------------------- */
#define SF_MAX_TENSORS_PER_LAUNCH 48

sf_status sf_adamw_layer_step(const sf_tensor* tensors, int n_tensors,
                              const sf_adamw_hparams* hp, int64_t step,
                              void* stream);

/* The same AdamW layer step on the host CPU cores, for layers whose arrays
 * are in host memory (any host memory; pinned is not required): SlideFormer's
 * own placement of the update (technical summary section 2.A, "the CPU
 * updates the parameters of layer L_i"), kept as a comparison point for the
 * device kernels.  Identical arithmetic to sf_adamw_layer_step (no
 * floating-point contraction, the same fused multiply-adds), so IEEE hosts
 * produce the same bits as the GPU for finite inputs.  n_threads <= 0 uses
 * one thread per core this process may run on (its CPU affinity set).
 * Synchronous: returns when the update is done. */
sf_status sf_adamw_host_step(const sf_tensor* tensors, int n_tensors,
                             const sf_adamw_hparams* hp, int64_t step,
                             int n_threads);

/* ------------------------------------------------------------------------
 * (b) Learned sparse projectors.
 *
 * A projector is a rows x d sparse matrix with exactly k entries in every
 * row, given as ELL: col_idx int32 [rows][k] (ids in [0, d)), val fp32
 * [rows][k], both device arrays, read once.  lsp_projector_create builds on
 * the device, in the stream, the library-owned index structures the kernels
 * use: the column lists of the transpose (CSC; rows ascending inside every
 * column, built by a stable counting sort), and the column order grouped by
 * list length (bucket 0 = empty column, else ceil(log2 nnz)+1; ascending
 * id inside a bucket).  The ELL arrays may be freed after the call returns
 * and the stream has passed it.
 *
 * `validate` != 0 checks on the device that every id is in [0, d) and that
 * no row repeats an id; a failed check makes the call return
 * SF_ERR_INVALID (the call then synchronises the stream).  With validate = 0
 * out-of-range ids are undefined behaviour and repeated ids add up.
 * Limits: 1 <= d <= 1024, 1 <= k <= 64, rows * k < 2^31.
 * ---------------------------------------------------------------------- */
typedef struct lsp_projector_s* lsp_projector;

sf_status lsp_projector_create(int64_t rows, int32_t d, int32_t k,
                               const int32_t* d_col_idx, const float* d_val,
                               int validate, void* stream, lsp_projector* out);

/* Copy the CSC and the bucket order out (device buffers, caller-owned):
 * col_ptr int32 [d+1], row_idx int32 [rows*k], val fp32 [rows*k],
 * bucket_perm int32 [d].  Any pointer may be NULL to skip that array. */
sf_status lsp_projector_export_csc(lsp_projector p, int32_t* col_ptr,
                                   int32_t* row_idx, float* val,
                                   int32_t* bucket_perm, void* stream);

/* Shape queries (return -1 for a NULL handle). */
int64_t lsp_projector_rows(lsp_projector p);
int32_t lsp_projector_dim(lsp_projector p);
int32_t lsp_projector_nnz_per_row(lsp_projector p);

/* Frees the handle.  The caller must make sure no enqueued work still uses
 * it (for example by synchronising its streams first). */
sf_status lsp_projector_destroy(lsp_projector p);

/* Bytes of device workspace that lsp_compress / lsp_decompress_apply need
 * for an m x n gradient and dimension d (the d x n or n x d intermediate). */
size_t lsp_workspace_bytes(int64_t m, int64_t n, int32_t d);

/* S = P^T G Q.
 *   P : projector with rows = m;  Q : projector with rows = n; same d.
 *   G : device, [m][n], dtype g_dtype (SF_BF16 or SF_FP32), row-major.
 *   S : device fp32 [d][d], written (S[a][c], a = column of P, c = column of Q).
 *   ws: device scratch of ws_bytes >= lsp_workspace_bytes(m, n, d).
 * fp32 accumulation; no atomics.  m, n >= 1. */
sf_status lsp_compress(lsp_projector P, lsp_projector Q, const void* G,
                       sf_dtype g_dtype, int64_t m, int64_t n, float* S,
                       void* ws, size_t ws_bytes, void* stream);

/* The matrices of one layer compressed in one call: S_i = P_i^T G_i Q_i for
 * i < count, the same results, bit for bit, as count lsp_compress calls
 * (every tile is computed as in its own launch).  The first stages of all
 * matrices whose G has one element type run in one launch, matrices with
 * the most row windows first, then all second stages in one launch, so the
 * GPU is filled across the layer's matrices instead of once per matrix (the
 * pages apply the projector step to every weight matrix of a layer).
 *   P, Q, G, g_dtype, m, n, S : arrays of count entries (host memory), each
 *       entry as the same argument of lsp_compress; every projector has the
 *       same d.
 *   ws : device scratch, 256-byte aligned, at least
 *       lsp_compress_layer_workspace_bytes(count, m, n, d) bytes (the
 *       matrices' compress workspaces one after another); the caller owns it.
 * Errors: SF_ERR_INVALID for count < 1, a NULL array or entry, rows that do
 * not match m or n, projectors of different d, a small or misaligned
 * workspace; otherwise as lsp_compress.  Asynchronous on `stream`. */
size_t lsp_compress_layer_workspace_bytes(int count, const int64_t* m,
                                          const int64_t* n, int32_t d);
sf_status lsp_compress_layer(int count, const lsp_projector* P,
                             const lsp_projector* Q, const void* const* G,
                             const int32_t* g_dtype, const int64_t* m,
                             const int64_t* n, float* const* S, void* ws,
                             size_t ws_bytes, void* stream);

/* lsp_compress for callers that cannot allocate device memory or hand the
 * library a workspace: callers under a framework whose caching allocator owns
 * the device memory pool, latency-critical loops where cudaMalloc's implicit
 * device-wide synchronisation is not acceptable, and thin bindings without an
 * allocator.  The papers have no counterpart; this is a library convenience.
 *
 * Same arguments, result and errors as lsp_compress, minus the workspace:
 * the intermediate lives in a fixed array of SF_NOALLOC_SCRATCH_BYTES that
 * is part of the library image (every GPU that loads the library holds it
 * until the process exits).  The call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *  - Shapes whose lsp_workspace_bytes(m, n, d) exceeds the array are
 *    rejected with SF_ERR_UNSUPPORTED and a message (for example
 *    d = 512 covers n up to 14,640 columns for any m).
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress), so the address stays right after a device
 *    reset; the first call on a device may also load the library's device
 *    code there, so make that first call before any stream capture.
 *  - Every call, on any stream, shares the one array, which keeps the last
 *    call's contents: calls that overlap on the GPU race and give undefined
 *    results.  Serialise them (one stream, or events).  Nothing in the
 *    array needs to start at zero. */
#define SF_NOALLOC_SCRATCH_BYTES (32u << 20)

sf_status lsp_compress_noalloc(lsp_projector P, lsp_projector Q, const void* G,
                               sf_dtype g_dtype, int64_t m, int64_t n, float* S,
                               void* stream);

/* AdamW in the compressed space, no weight decay, step t = `step` >= 1:
 *   m  <- beta1*m + (1-beta1)*S;  v <- beta2*v + (1-beta2)*S^2
 *   dS  = (lr/(1-beta1^t)) * m / (sqrt(v)/sqrt(1-beta2^t) + eps)
 * S, m, v, dS: device fp32 [d2] (d2 = d*d; any element count works).
 * hp->weight_decay is ignored. */
sf_status lsp_adamw_compressed(const float* S, float* m, float* v, float* dS,
                               int64_t d2, const sf_adamw_hparams* hp,
                               int64_t step, void* stream);

/* W <- W - P dS Q^T.
 *   dS : device fp32 [d][d] (same layout as S).
 *   W  : device [m][n], dtype w_dtype: SF_FP32 (an fp32 master: W - D in
 *        fp32) or SF_BF16 (bf16 weights: RNE(float(W) - D)).
 *   w_bf16_mirror: NULL, or device bf16 [m][n] that receives RNE of the new
 *        fp32 W (only with w_dtype = SF_FP32).
 *   ws : device scratch, as for lsp_compress.
 * No weight decay is applied here. */
sf_status lsp_decompress_apply(lsp_projector P, lsp_projector Q, const float* dS,
                               void* W, sf_dtype w_dtype, void* w_bf16_mirror,
                               int64_t m, int64_t n, void* ws, size_t ws_bytes,
                               void* stream);

/* Learning the projectors (LSP-Offload, method section, "key design": the
 * sparse projectors are fitted by gradient descent to minimise what is lost
 * by compressing and decompressing).  The pages give no loss or schedule;
 * this is one plain gradient step on the stored values of P and Q (their
 * column ids stay fixed) for the squared reconstruction error of a gradient
 * sample G:
 *
 *   S = P^T G Q,   L = || G - P S Q^T ||_F^2,
 *   dL/dP = -2 (E Q S^T + G Q Q^T E^T P),  dL/dQ = -2 (E^T P S + G^T P P^T E Q),
 *   E = G - P S Q^T,   val <- val - lr * dL/dval   (P and Q together, both
 *   gradients at the values before the step).
 *
 *   P, Q   : projectors with rows m and n, the same d; must be different
 *            handles, and neither may have had out-of-range column ids at
 *            creation (SF_ERR_INVALID otherwise).  Their values are updated
 *            in place, in every layout the library keeps, so later
 *            compress / decompress calls and exports see the new values.
 *   G      : device, [m][n] row-major, SF_BF16 or SF_FP32.
 *   lr     : step size (rounded once to fp32); lr = 0 evaluates only.
 *   loss   : device double [1], receives L before the step; may be NULL.
 *   grad_P : device fp32 [m * k_P], receives dL/dval of P in ELL order (row
 *            i, entry t at i * k_P + t); may be NULL.  grad_Q likewise
 *            [n * k_Q].
 *   ws     : device scratch of ws_bytes >= lsp_fit_workspace_bytes(m, n, d,
 *            g_dtype), 256-byte aligned.
 * fp32 arithmetic (the loss assembled in fp64 from fp32 partial sums); no
 * atomics; stream-ordered like every other call. */
size_t lsp_fit_workspace_bytes(int64_t m, int64_t n, int32_t d, sf_dtype g_dtype);

sf_status lsp_projector_fit_step(lsp_projector P, lsp_projector Q, const void* G,
                                 sf_dtype g_dtype, int64_t m, int64_t n, double lr,
                                 double* loss, float* grad_P, float* grad_Q,
                                 void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Dense products on the tensor cores (building block of the fused linear
 * cross-entropy below; usable on its own).
 *
 * C = alpha * A * B^T            (accumulate = 0)
 * C = C + alpha * A * B^T        (accumulate = 1)
 *   A : device bf16 [M][lda], row-major, the first K columns used.
 *   B : device bf16 [N][ldb], row-major, the first K columns used.
 *   C : device fp32 [M][ldc], row-major.
 * bf16 products accumulated in fp32 on the tensor cores (tcgen05.mma).
 * A and B need 16-byte aligned bases and lda, ldb multiples of 8
 * (SF_ERR_UNSUPPORTED otherwise); M, N, K >= 1; no other shape limits.
 * Deterministic for a given shape. */
sf_status sf_gemm_abt_bf16(const void* A, const void* B, float* C, int64_t M,
                           int64_t N, int64_t K, int64_t lda, int64_t ldb,
                           int64_t ldc, float alpha, int accumulate, void* stream);

/* The same product with either operand stored transposed:
 *   a_layout 0: A is [M][lda] row-major (K-major), lda >= K;
 *   a_layout 1: A is stored as A^T, [K][lda] row-major (M-major), lda >= M;
 *   b_layout 0: B is [N][ldb] row-major (K-major), ldb >= K;
 *   b_layout 1: B is stored as B^T, [K][ldb] row-major (N-major), ldb >= N.
 * For example, b_layout 1 with a row-major X [K][N] as B gives
 * C = alpha * A * X, and a_layout 1 with a row-major Y [K][M] as A gives
 * C = alpha * Y^T * B^T.  A layout other than 0 or 1 returns SF_ERR_INVALID;
 * alignment, shape limits and determinism as sf_gemm_abt_bf16 (which is
 * layouts 0, 0). */
sf_status sf_gemm_bf16(const void* A, int a_layout, const void* B, int b_layout,
                       float* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldc, float alpha, int accumulate,
                       void* stream);

/* ------------------------------------------------------------------------
 * Fused linear cross-entropy (SlideFormer, "Fused LinearCrossEntropy" in the
 * summaries' kernel lists: the output projection and the loss fused, the
 * gradients computed in small blocks so the full logits tensor is never
 * held).  For hidden states H (N tokens x D) and an output layer W (V x D):
 *
 *   z_i  = W h_i,   n = number of tokens whose label != ignore_index
 *   loss = (1/n) sum_{labelled i} ( logsumexp(z_i) - z_i[label_i] )
 *   dH   = dZ W,   dW = dZ^T H,   dZ_i = (softmax(z_i) - onehot(label_i)) / n
 *          (dZ_i = 0 for unlabelled tokens; loss = 0 and no gradient if n = 0)
 *
 *   H      : device bf16 [N][D] row-major;  W : device bf16 [V][D] row-major.
 *   labels : device int32 [N]; a label outside [0, V) that is not
 *            ignore_index counts as unlabelled and is reported by
 *            sf_sync_status (SF_ERR_INVALID).
 *   chunk  : tokens per block (a positive multiple of 8; the call holds one
 *            chunk of fp32 logits and one of the bf16 gradient, no
 *            transposed copies).
 *   loss   : device double [1], written; may be NULL.
 *   dH     : device fp32 [N][D], written; may be NULL.
 *   dW     : device fp32 [V][D], written; may be NULL (both NULL: loss only).
 *   ws     : device scratch of ws_bytes >= lce_workspace_bytes(N, D, V,
 *            chunk), 256-byte aligned.
 * Logits: bf16 products summed in fp32 on the tensor cores.  The row
 * statistics are fp32; dZ is rounded to bf16 (nearest even) before the two
 * gradient products, which run on the tensor cores with fp32 sums.
 * D and V must be multiples of 8 and H, W, dH, dW 16-byte aligned
 * (SF_ERR_UNSUPPORTED otherwise).  Deterministic. */
size_t lce_workspace_bytes(int64_t n_tokens, int64_t d, int64_t vocab, int64_t chunk);

sf_status lce_forward_backward(const void* H, const void* W, const int32_t* labels,
                               int64_t N, int64_t D, int64_t V, int64_t chunk,
                               int32_t ignore_index, double* loss, float* dH,
                               float* dW, void* ws, size_t ws_bytes, void* stream);

/* Copy a projector's current values, ELL order [rows * k] fp32, to device
 * memory `val` (after lsp_projector_fit_step they differ from the values
 * the projector was created with).  Out-of-range ids read as 0. */
sf_status lsp_projector_export_values(lsp_projector p, float* val, void* stream);

/* ------------------------------------------------------------------------
 * (c) Layer-sliding window.
 *
 * A window owns n_slots (>= 1) caller-allocated device slots.  Each slot is
 * an array of sf_tensor holding device buffers big enough for the largest
 * layer that will pass through it (tensor i of a slot must have numel >=
 * tensor i of every layer).  The window creates its own CUDA events; it
 * uses the three caller streams: h2d (host -> device copies), compute (the
 * AdamW kernel), d2h (device -> host copies).
 *
 * sf_slide_window_step enqueues, for every entry l = order[v] in turn
 * (v = 0..n_order-1), with slot s = v mod n_slots:
 *   h2d:     wait until slot s is free and layer l's previous write-back
 *            has landed; copy grad, master, exp_avg, exp_avg_sq of layer l
 *            (pinned host) into slot s;
 *   compute: wait for the copies; run sf_adamw_layer_step on slot s with
 *            step = ++steps[l];
 *   d2h:     wait for the update; copy master, exp_avg, exp_avg_sq and
 *            weight (if the host layer has one) back to layer l; the slot is
 *            free again when these copies end.
 * Copies are issued per array (grad, master, exp_avg, exp_avg_sq, weight):
 * consecutive tensors whose host arrays and slot arrays both follow one
 * another in memory move as one copy (a layer kept as flat per-array
 * buffers moves as one copy per array); the bytes moved are the same.
 * Host-layer pointers must be pinned (page-locked) host memory, except that
 * any array of a layer may instead be device memory of the current device
 * (for instance fp32 master weights and moments kept resident in HBM while
 * gradients come from and bf16 weights go back to pinned host memory): such
 * an array is updated in place, is neither copied in nor written back, and
 * the slot's buffer for it is not used and may be NULL (a slot buffer may be
 * NULL only for arrays that every layer passing through keeps in device
 * memory; SF_ERR_INVALID otherwise).  The call returns when everything is
 * enqueued; `steps` (int64 [n_layers], host) is updated on return.  Host
 * buffers of a layer must not be touched until its copies have ended
 * (sf_window_sync).
 * ---------------------------------------------------------------------- */
typedef struct sf_window_s* sf_window;

typedef struct {
  const sf_tensor* tensors; /* pinned host pointers */
  int n_tensors;
} sf_host_layer;

sf_status sf_window_create(int n_slots, const sf_tensor* const* device_slots,
                           int n_tensors_per_slot, void* h2d_stream,
                           void* compute_stream, void* d2h_stream,
                           sf_window* out);

sf_status sf_slide_window_step(sf_window w, const sf_host_layer* layers,
                               int n_layers, const int32_t* order, int n_order,
                               const sf_adamw_hparams* hp, int64_t* steps);

/* Waits, with a bound, until all work the window enqueued has ended.
 * timeout_ms <= 0 uses the default bound (SF_TIMEOUT_MS environment
 * variable, else 600000 ms).  Returns SF_ERR_TIMEOUT when the bound runs
 * out (the work is still in flight; the window stays usable). */
sf_status sf_window_sync(sf_window w, int64_t timeout_ms);

/* Frees the window's events.  Waits (bounded) for its work first. */
sf_status sf_window_destroy(sf_window w);

/* ------------------------------------------------------------------------
 * (b') Learned sparse projectors with the compressed optimizer state in
 * pinned host memory, layer by layer.
 *
 * LSP-Offload ("Practical offloading for fine-tuning LLM on commodity GPU
 * via learned sparse projectors", abstract: "layer-wise communication
 * schedule") keeps only compressed d x d quantities on the host and
 * overlaps their transfers with the compute of neighbouring layers.  Here
 * each layer's compressed moments m~, v~ (fp32 [d][d]) live in pinned host
 * memory; lsp_slide_window_step enqueues, for every entry l = order[v]
 * (slot s = running visit count mod n_slots):
 *   compute: lsp_compress(P, Q, G) -> slot S           (device)
 *   h2d:     wait until slot s is free and layer l's previous write-back has
 *            landed; copy m~, v~ of layer l into the slot
 *   compute: lsp_adamw_compressed(S, m~, v~ -> dS, step = ++steps[l]);
 *            lsp_decompress_apply(P, Q, dS, W)
 *   d2h:     copy m~, v~ back to layer l; the slot is free again when these
 *            copies have ended.
 * Results are bitwise those of the same calls with device-resident moments.
 * Slots are caller-allocated device buffers; the window owns only events.
 * ---------------------------------------------------------------------- */
typedef struct {
  float* S;       /* device fp32 [d][d] */
  float* m;       /* device fp32 [d][d] */
  float* v;       /* device fp32 [d][d] */
  float* dS;      /* device fp32 [d][d] */
  void* ws;       /* device workspace (256-byte aligned) */
  size_t ws_bytes;
} lsp_slot;

typedef struct {
  lsp_projector P;      /* rows = m */
  lsp_projector Q;      /* rows = n, same d as P */
  const void* G;        /* device [m][n], dtype g_dtype */
  sf_dtype g_dtype;
  void* W;              /* device [m][n], dtype w_dtype */
  sf_dtype w_dtype;
  void* w_bf16_mirror;  /* NULL or device bf16 [m][n] (w_dtype = SF_FP32) */
  int64_t m, n;
  float* m_host;        /* pinned host fp32 [d][d]: compressed first moment */
  float* v_host;        /* pinned host fp32 [d][d]: compressed second moment */
} lsp_layer;

typedef struct lsp_window_s* lsp_window;

/* n_slots >= 1 slots of dimension d; every slot's ws must cover every layer
 * that passes through (lsp_workspace_bytes). */
sf_status lsp_window_create(int n_slots, const lsp_slot* slots, int32_t d,
                            void* h2d_stream, void* compute_stream,
                            void* d2h_stream, lsp_window* out);

sf_status lsp_slide_window_step(lsp_window w, const lsp_layer* layers,
                                int n_layers, const int32_t* order, int n_order,
                                const sf_adamw_hparams* hp, int64_t* steps);

/* The same window with the compressed AdamW on the host cores, LSP-Offload's
 * own placement of the update (method section: the CPU computes in the
 * compressed space; abstract: layer-wise communication schedule).  For every
 * entry l = order[u] (slot s = running visit count mod n_slots):
 *   compute: lsp_compress(P, Q, G) -> slot S           (device)
 *   d2h:     S -> slot S_host (pinned host)
 *   host:    a host function ordered after that copy runs the compressed
 *            AdamW (step = ++steps[l], no weight decay) on the host cores on
 *            m_host, v_host of layer l in place, writing dS to slot dS_host
 *   h2d:     dS_host -> slot dS                           (device)
 *   compute: lsp_decompress_apply(P, Q, dS, W)
 * The compress of the next n_slots - 1 visits is enqueued before a visit's
 * decompress-apply, so a layer's host round trip overlaps the next layers'
 * GPU work (n_slots >= 2 for any overlap).  Per layer the host link carries
 * S down and dS up (d*d*4 bytes each way) and no moments.  The host
 * arithmetic is the device kernel's (same operations, same order, no
 * floating-point contraction), so results are bitwise those of
 * lsp_adamw_compressed on device-resident moments.
 *   n_threads: host threads of the update (<= 0: up to 8 of the cores this
 *   process may run on); the window starts them here and stops them in
 *   lsp_window_destroy.
 * lsp_slide_window_step, lsp_window_sync and lsp_window_destroy take either
 * kind of window.  The m_host / v_host of a layer and the host staging
 * buffers must not be touched until lsp_window_sync has returned. */
typedef struct {
  float* S;        /* device fp32 [d][d] */
  float* dS;       /* device fp32 [d][d] */
  float* S_host;   /* pinned host fp32 [d][d]: S on its way to the host update */
  float* dS_host;  /* pinned host fp32 [d][d]: dS on its way back */
  void* ws;        /* device workspace (256-byte aligned) */
  size_t ws_bytes;
} lsp_host_slot;

sf_status lsp_window_create_host_update(int n_slots, const lsp_host_slot* slots,
                                        int32_t d, int n_threads,
                                        void* h2d_stream, void* compute_stream,
                                        void* d2h_stream, lsp_window* out);

/* Measurement hook of a host-update window: a timeline of its visits.
 * lsp_window_timeline_start waits for the window's work, then makes the
 * next `capacity` visits (over any number of lsp_slide_window_step calls)
 * record 9 timing events each; capacity 0 switches it off.
 * lsp_window_timeline_read waits for the window's work and writes, for up
 * to `capacity` recorded visits in visit order, 9 floats per visit into
 * `ms` (host), milliseconds after the first visit's first point: compress
 * start and end (compute stream), S-to-host copy start and end and host
 * update end (d2h stream; the update starts when the copy ends), dS copy
 * start and end (h2d stream), decompress-apply start and end (compute
 * stream); *n_visits = the visits written.  Overlap shows as one visit's
 * copies and host update lying inside other visits' compress and
 * decompress-apply.  SF_ERR_INVALID for a device-update window, a NULL
 * pointer or a capacity outside [0, 2^20]. */
sf_status lsp_window_timeline_start(lsp_window w, int capacity);
sf_status lsp_window_timeline_read(lsp_window w, float* ms, int capacity, int* n_visits);

/* Bounded wait (as sf_window_sync) for everything the window enqueued. */
sf_status lsp_window_sync(lsp_window w, int64_t timeout_ms);

/* Waits (bounded) for the window's work, then frees its events and host
 * threads.  If the wait runs out (SF_ERR_TIMEOUT) the window is kept, since
 * work still in flight may use it; call lsp_window_destroy again later. */
sf_status lsp_window_destroy(lsp_window w);

/* ------------------------------------------------------------------------
 * Utilities.
 * ---------------------------------------------------------------------- */

/* Waits, with the default bound, for `stream` and returns SF_OK or the
 * sticky error of the CUDA context (SF_ERR_CUDA), or SF_ERR_TIMEOUT. */
sf_status sf_sync_status(void* stream);

/* Message for the calling thread's last failed call ("" if none). */
const char* sf_last_error(void);

/* Library version, e.g. "0.1.0". */
const char* sf_version(void);

/* Test hook for failure handling: the n-th host->device or device->host
 * copy that a window enqueues after this call fails once on the host, before
 * anything is handed to CUDA, and the window call returns SF_ERR_CUDA with
 * the message "injected copy failure".  n = 0 switches the hook off.  Not
 * thread-safe; meant for tests only. */
void sf_test_fail_copy_after(int64_t n);

/* Test hook for the kernels' bounded waits: launches one warp that waits on
 * an mbarrier nothing arrives on, with a limit of limit_cycles SM clock
 * cycles (1 .. 4e9; the library's own waits use ~4e9, about 2 s).  The wait
 * runs out, records the timeout in the device error word and the kernel
 * returns, so the next sf_sync_status() returns SF_ERR_TIMEOUT and clears
 * it; the context stays usable.  SF_ERR_INVALID for a limit out of range. */
sf_status sf_test_device_wait_runs_out(int64_t limit_cycles, void* stream);

/* Measurement hook: the shared-memory gather rate that bounds the projector
 * kernels (compress and decompress are sparse products whose every
 * multiply-add reads a shared-memory tile row chosen by a projector index).
 * Launches `ctas` CTAs of 512 threads; each thread runs `iters` steps of the
 * gather kernels' inner loop (two entries, two 16-byte tile loads at dynamic
 * rows, 8 fp32 multiply-adds) on shared-memory data only, and writes one
 * float to sink[cta * 512 + thread] (device, ctas * 512 floats) so the work
 * is not optimised away.  Multiply-adds done: ctas * 512 * iters * 8; the
 * caller times the call (CUDA events on `stream`).  SF_ERR_INVALID for
 * ctas < 1, iters < 1 or a NULL sink. */
sf_status sf_bench_gather_rate(int32_t ctas, int64_t iters, float* sink, void* stream);

/* Measurement hook: the tensor-memory (TMEM) gather rate, another
 * on-chip roof for the projector kernels (LSP-Offload, method
 * section: the compress and decompress are sparse products whose dense
 * operand is read at rows chosen by projector indices).  Launches `ctas`
 * CTAs of 512 threads, one per SM, each allocating all 512 TMEM columns for
 * the duration of the launch (released before it ends).  Every thread runs
 * `iters` steps; a step issues 8 tcgen05.ld.32x32b loads of `x` (1, 2 or 4)
 * consecutive 32-bit columns of its lane at columns chosen per load, waits
 * for them and does 8 * x fp32 multiply-adds.  With `entries` != 0 each
 * load's column and multiplier come from an 8-byte entry in shared memory
 * (as in a gather kernel), else they are computed in registers.  Writes one
 * float to sink[cta * 512 + thread] (device, ctas * 512 floats).
 * Multiply-adds done: ctas * 512 * iters * 8 * x; the caller times the call
 * (CUDA events on `stream`).  SF_ERR_INVALID for ctas < 1, iters < 1, a NULL
 * sink or x not in {1, 2, 4}. */
sf_status sf_bench_tmem_rate(int32_t ctas, int64_t iters, int32_t x, int32_t entries, float* sink, void* stream);

/* Measurement hook: the rate of row gathers served from L2 (the source a
 * gather reads when its dense operand is not staged on chip).  `buf` is a
 * device array of `rows` rows of 128 floats (512 bytes, 16-byte aligned);
 * launches `ctas` CTAs of 256 threads; each warp runs `iters` steps of 16
 * row loads (one 16-byte load per lane, rows chosen by a per-warp
 * generator, all 16 in flight) followed by 64 multiply-adds per lane, and
 * each thread writes one float to sink[cta * 256 + thread] (device, ctas *
 * 256 floats).  Bytes gathered: ctas * 8 * iters * 16 * 512.  With
 * rows * 512 bytes well below L2's size and the buffer read once before,
 * the loads hit L2.  SF_ERR_INVALID for ctas, iters or rows below 1, rows
 * of 2^32 or more, NULL pointers or an unaligned buf. */
sf_status sf_bench_l2_gather_rate(int32_t ctas, int64_t iters, const float* buf, int64_t rows, float* sink,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SFOPT_H */

"""Thin ctypes binding over the C ABI of ``libsfopt.so`` (include/sfopt.h).

Argument marshalling only: every step of the update runs in the library's
CUDA kernels.  Functions keep the C names; they take torch tensors (or raw
integer addresses), torch CUDA streams and plain Python numbers, and raise
``SfError`` when the library returns a non-OK status.  There is no fallback:
if the library is missing or fails to load, ``load()`` raises.
"""

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libsfopt.so")

SF_OK, SF_ERR_INVALID, SF_ERR_CUDA, SF_ERR_OOM, SF_ERR_UNSUPPORTED, SF_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
SF_BF16, SF_FP32 = 0, 1
SF_MAX_TENSORS_PER_LAUNCH = 48

# Every symbol include/sfopt.h declares.
EXPORTS = [
    "sf_adamw_layer_step", "lsp_projector_create", "lsp_projector_export_csc",
    "lsp_projector_rows", "lsp_projector_dim", "lsp_projector_nnz_per_row",
    "lsp_projector_destroy", "lsp_workspace_bytes", "lsp_compress", "lsp_adamw_compressed",
    "lsp_decompress_apply", "sf_window_create", "sf_slide_window_step", "sf_window_sync",
    "sf_window_destroy", "sf_sync_status", "sf_last_error", "sf_version",
    "sf_test_fail_copy_after", "lsp_compress_noalloc", "lsp_compress_layer_workspace_bytes", "lsp_compress_layer",
    "lsp_window_create", "lsp_slide_window_step", "lsp_window_sync", "lsp_window_destroy",
    "lsp_window_create_host_update", "lsp_window_timeline_start", "lsp_window_timeline_read",
    "sf_adamw_host_step", "lsp_fit_workspace_bytes", "lsp_projector_fit_step", "lsp_projector_export_values",
    "sf_gemm_abt_bf16", "sf_gemm_bf16", "sf_bench_gather_rate", "sf_bench_tmem_rate", "sf_bench_l2_gather_rate",
    "lce_workspace_bytes", "lce_forward_backward",
    "sf_test_device_wait_runs_out",
]


class SfError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"status {status}: {msg}")
        self.status = status


class sf_adamw_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double)]


class sf_tensor(ctypes.Structure):
    _fields_ = [("grad", ctypes.c_void_p), ("master", ctypes.c_void_p), ("exp_avg", ctypes.c_void_p),
                ("exp_avg_sq", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("numel", ctypes.c_int64)]


class sf_host_layer(ctypes.Structure):
    _fields_ = [("tensors", ctypes.POINTER(sf_tensor)), ("n_tensors", ctypes.c_int)]


class lsp_host_slot(ctypes.Structure):
    _fields_ = [("S", ctypes.c_void_p), ("dS", ctypes.c_void_p), ("S_host", ctypes.c_void_p),
                ("dS_host", ctypes.c_void_p), ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t)]


class lsp_slot(ctypes.Structure):
    _fields_ = [("S", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dS", ctypes.c_void_p),
                ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t)]


class lsp_layer(ctypes.Structure):
    _fields_ = [("P", ctypes.c_void_p), ("Q", ctypes.c_void_p), ("G", ctypes.c_void_p), ("g_dtype", ctypes.c_int),
                ("W", ctypes.c_void_p), ("w_dtype", ctypes.c_int), ("w_bf16_mirror", ctypes.c_void_p),
                ("m", ctypes.c_int64), ("n", ctypes.c_int64), ("m_host", ctypes.c_void_p),
                ("v_host", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_INT = ctypes.c_int
_ST = ctypes.c_int

_SIGS = {
    "sf_adamw_layer_step": (_ST, [ctypes.POINTER(sf_tensor), _INT, ctypes.POINTER(sf_adamw_hparams), _I64, _P]),
    "lsp_projector_create": (_ST, [_I64, _I32, _I32, _P, _P, _INT, _P, ctypes.POINTER(_P)]),
    "lsp_projector_export_csc": (_ST, [_P, _P, _P, _P, _P, _P]),
    "lsp_projector_rows": (_I64, [_P]),
    "lsp_projector_dim": (_I32, [_P]),
    "lsp_projector_nnz_per_row": (_I32, [_P]),
    "lsp_projector_destroy": (_ST, [_P]),
    "lsp_workspace_bytes": (ctypes.c_size_t, [_I64, _I64, _I32]),
    "lsp_compress": (_ST, [_P, _P, _P, _INT, _I64, _I64, _P, _P, ctypes.c_size_t, _P]),
    "lsp_compress_noalloc": (_ST, [_P, _P, _P, _INT, _I64, _I64, _P, _P]),
    "lsp_compress_layer_workspace_bytes": (ctypes.c_size_t, [_INT, _P, _P, ctypes.c_int32]),
    "lsp_compress_layer": (_ST, [_INT, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "lsp_adamw_compressed": (_ST, [_P, _P, _P, _P, _I64, ctypes.POINTER(sf_adamw_hparams), _I64, _P]),
    "lsp_decompress_apply": (_ST, [_P, _P, _P, _P, _INT, _P, _I64, _I64, _P, ctypes.c_size_t, _P]),
    "sf_window_create": (_ST, [_INT, ctypes.POINTER(ctypes.POINTER(sf_tensor)), _INT, _P, _P, _P, ctypes.POINTER(_P)]),
    "sf_slide_window_step": (_ST, [_P, ctypes.POINTER(sf_host_layer), _INT, ctypes.POINTER(_I32), _INT,
                                   ctypes.POINTER(sf_adamw_hparams), ctypes.POINTER(_I64)]),
    "sf_window_sync": (_ST, [_P, _I64]),
    "sf_window_destroy": (_ST, [_P]),
    "sf_sync_status": (_ST, [_P]),
    "sf_last_error": (ctypes.c_char_p, []),
    "sf_version": (ctypes.c_char_p, []),
    "sf_test_fail_copy_after": (None, [_I64]),
    "sf_adamw_host_step": (_ST, [ctypes.POINTER(sf_tensor), _INT, ctypes.POINTER(sf_adamw_hparams), _I64, _INT]),
    "lsp_window_create": (_ST, [_INT, ctypes.POINTER(lsp_slot), _I32, _P, _P, _P, ctypes.POINTER(_P)]),
    "lsp_window_create_host_update": (_ST, [_INT, ctypes.POINTER(lsp_host_slot), _I32, _INT, _P, _P, _P,
                                            ctypes.POINTER(_P)]),
    "lsp_window_timeline_start": (_ST, [_P, _INT]),
    "lsp_window_timeline_read": (_ST, [_P, _P, _INT, ctypes.POINTER(_INT)]),
    "lsp_slide_window_step": (_ST, [_P, ctypes.POINTER(lsp_layer), _INT, ctypes.POINTER(_I32), _INT,
                                    ctypes.POINTER(sf_adamw_hparams), ctypes.POINTER(_I64)]),
    "lsp_window_sync": (_ST, [_P, _I64]),
    "lsp_window_destroy": (_ST, [_P]),
    "lsp_fit_workspace_bytes": (ctypes.c_size_t, [_I64, _I64, _I32, _INT]),
    "lsp_projector_fit_step": (_ST, [_P, _P, _P, _INT, _I64, _I64, ctypes.c_double, _P, _P, _P, _P,
                                     ctypes.c_size_t, _P]),
    "lsp_projector_export_values": (_ST, [_P, _P, _P]),
    "sf_gemm_abt_bf16": (_ST, [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, ctypes.c_float, _INT, _P]),
    "sf_bench_gather_rate": (_ST, [_INT, _I64, _P, _P]),
    "sf_bench_tmem_rate": (_ST, [_INT, _I64, _INT, _INT, _P, _P]),
    "sf_bench_l2_gather_rate": (_ST, [_INT, _I64, _P, _I64, _P, _P]),
    "sf_gemm_bf16": (_ST, [_P, _INT, _P, _INT, _P, _I64, _I64, _I64, _I64, _I64, _I64, ctypes.c_float, _INT, _P]),
    "lce_workspace_bytes": (ctypes.c_size_t, [_I64, _I64, _I64, _I64]),
    "sf_test_device_wait_runs_out": (_ST, [_I64, _P]),
    "lce_forward_backward": (_ST, [_P, _P, _P, _I64, _I64, _I64, _I64, _I32, _P, _P, _P, _P, ctypes.c_size_t, _P]),
}

_lib = None


def load(path=None):
    """Load libsfopt.so (built by ``layer_optimizer_gb300.build``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with `python -m layer_optimizer_gb300.build`")
    try:  # make sure a libcudart with the library's SONAME is in the process (torch ships one)
        import torch  # noqa: F401
    except ImportError:
        pass
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(st):
    if st != SF_OK:
        raise SfError(st, load().sf_last_error().decode())


def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def hparams(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01):
    return sf_adamw_hparams(lr, beta1, beta2, eps, weight_decay)


def make_tensor(grad, master, exp_avg, exp_avg_sq, weight=None, numel=None):
    """sf_tensor from torch tensors (or addresses; then ``numel`` is required)."""
    n = numel if numel is not None else master.numel()
    return sf_tensor(_addr(grad), _addr(master), _addr(exp_avg), _addr(exp_avg_sq), _addr(weight), n)


def tensor_array(items):
    arr = (sf_tensor * max(1, len(items)))()
    for i, t in enumerate(items):
        arr[i] = t if isinstance(t, sf_tensor) else make_tensor(*t)
    return arr


# ------------------------------------------------------------------ (a) ----

def sf_adamw_layer_step(tensors, hp, step, stream=None):
    arr = tensor_array(tensors)
    _check(load().sf_adamw_layer_step(arr, len(tensors), ctypes.byref(hp), step, _stream(stream)))


def sf_adamw_host_step(tensors, hp, step, n_threads=0):
    """The same update on the host cores; tensors hold host (CPU) arrays."""
    arr = tensor_array(tensors)
    _check(load().sf_adamw_host_step(arr, len(tensors), ctypes.byref(hp), step, n_threads))


# ------------------------------------------------------------------ (b) ----

class Projector:
    """Owning wrapper of an lsp_projector handle."""

    def __init__(self, handle):
        self.handle = handle

    @property
    def rows(self):
        return load().lsp_projector_rows(self.handle)

    @property
    def d(self):
        return load().lsp_projector_dim(self.handle)

    @property
    def k(self):
        return load().lsp_projector_nnz_per_row(self.handle)

    def close(self):
        if self.handle:
            _check(load().lsp_projector_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            if self.handle:
                load().lsp_projector_destroy(self.handle)
        except Exception:
            pass


def lsp_projector_create(rows, d, k, col_idx, val, validate=True, stream=None):
    h = ctypes.c_void_p()
    _check(load().lsp_projector_create(rows, d, k, _addr(col_idx), _addr(val), int(bool(validate)),
                                       _stream(stream), ctypes.byref(h)))
    return Projector(h.value)


def lsp_projector_export_csc(p, col_ptr=None, row_idx=None, val=None, bucket_perm=None, stream=None):
    _check(load().lsp_projector_export_csc(p.handle, _addr(col_ptr), _addr(row_idx), _addr(val),
                                           _addr(bucket_perm), _stream(stream)))


def lsp_workspace_bytes(m, n, d):
    return load().lsp_workspace_bytes(m, n, d)


def lsp_compress(P, Q, G, g_dtype, m, n, S, ws, ws_bytes, stream=None):
    _check(load().lsp_compress(P.handle, Q.handle, _addr(G), g_dtype, m, n, _addr(S), _addr(ws),
                               ws_bytes, _stream(stream)))


def lsp_compress_layer_workspace_bytes(ms, ns, d):
    c = len(ms)
    return load().lsp_compress_layer_workspace_bytes(c, (ctypes.c_int64 * c)(*ms), (ctypes.c_int64 * c)(*ns), d)


def lsp_compress_layer(Ps, Qs, Gs, g_dtypes, ms, ns, Ss, ws, ws_bytes, stream=None):
    """One layer's matrices in one call: lists of projectors, gradients, dtypes, sizes and outputs."""
    c = len(Ps)
    _check(load().lsp_compress_layer(c, (ctypes.c_void_p * c)(*[p.handle for p in Ps]),
                                     (ctypes.c_void_p * c)(*[q.handle for q in Qs]),
                                     (ctypes.c_void_p * c)(*[_addr(g) for g in Gs]),
                                     (ctypes.c_int32 * c)(*g_dtypes), (ctypes.c_int64 * c)(*ms),
                                     (ctypes.c_int64 * c)(*ns), (ctypes.c_void_p * c)(*[_addr(x) for x in Ss]),
                                     _addr(ws), ws_bytes, _stream(stream)))


def lsp_compress_noalloc(P, Q, G, g_dtype, m, n, S, stream=None):
    _check(load().lsp_compress_noalloc(P.handle, Q.handle, _addr(G), g_dtype, m, n, _addr(S), _stream(stream)))


SF_NOALLOC_SCRATCH_BYTES = 32 << 20


def lsp_adamw_compressed(S, m, v, dS, d2, hp, step, stream=None):
    _check(load().lsp_adamw_compressed(_addr(S), _addr(m), _addr(v), _addr(dS), d2, ctypes.byref(hp),
                                       step, _stream(stream)))


def lsp_decompress_apply(P, Q, dS, W, w_dtype, w_bf16_mirror, m, n, ws, ws_bytes, stream=None):
    _check(load().lsp_decompress_apply(P.handle, Q.handle, _addr(dS), _addr(W), w_dtype,
                                       _addr(w_bf16_mirror), m, n, _addr(ws), ws_bytes, _stream(stream)))


def lsp_fit_workspace_bytes(m, n, d, g_dtype):
    return load().lsp_fit_workspace_bytes(m, n, d, g_dtype)


def lsp_projector_fit_step(P, Q, G, g_dtype, m, n, lr, loss, grad_P, grad_Q, ws, ws_bytes, stream=None):
    _check(load().lsp_projector_fit_step(P.handle, Q.handle, _addr(G), g_dtype, m, n, float(lr), _addr(loss),
                                         _addr(grad_P), _addr(grad_Q), _addr(ws), ws_bytes, _stream(stream)))


def lsp_projector_export_values(p, val, stream=None):
    _check(load().lsp_projector_export_values(p.handle, _addr(val), _stream(stream)))


def sf_gemm_abt_bf16(A, B, C, M, N, K, lda, ldb, ldc, alpha=1.0, accumulate=False, stream=None):
    _check(load().sf_gemm_abt_bf16(_addr(A), _addr(B), _addr(C), M, N, K, lda, ldb, ldc, float(alpha),
                                   int(bool(accumulate)), _stream(stream)))


def sf_gemm_bf16(A, a_layout, B, b_layout, C, M, N, K, lda, ldb, ldc, alpha=1.0, accumulate=False, stream=None):
    _check(load().sf_gemm_bf16(_addr(A), int(a_layout), _addr(B), int(b_layout), _addr(C), M, N, K, lda, ldb, ldc,
                               float(alpha), int(bool(accumulate)), _stream(stream)))


def sf_bench_gather_rate(ctas, iters, sink, stream=None):
    _check(load().sf_bench_gather_rate(int(ctas), int(iters), _addr(sink), _stream(stream)))


def sf_bench_tmem_rate(ctas, iters, x, entries, sink, stream=None):
    _check(load().sf_bench_tmem_rate(int(ctas), int(iters), int(x), int(entries), _addr(sink), _stream(stream)))


def sf_bench_l2_gather_rate(ctas, iters, buf, rows, sink, stream=None):
    _check(load().sf_bench_l2_gather_rate(int(ctas), int(iters), _addr(buf), int(rows), _addr(sink),
                                          _stream(stream)))


def lce_workspace_bytes(n_tokens, d, vocab, chunk):
    return load().lce_workspace_bytes(n_tokens, d, vocab, chunk)


def lce_forward_backward(H, W, labels, N, D, V, chunk, ignore_index, loss, dH, dW, ws, ws_bytes, stream=None):
    _check(load().lce_forward_backward(_addr(H), _addr(W), _addr(labels), N, D, V, chunk, ignore_index, _addr(loss),
                                       _addr(dH), _addr(dW), _addr(ws), ws_bytes, _stream(stream)))


# ------------------------------------------------------------------ (c) ----

class Window:
    """Owning wrapper of an sf_window handle; keeps its slot arrays alive."""

    def __init__(self, handle, keep):
        self.handle = handle
        self._keep = keep

    def sync(self, timeout_ms=0):
        _check(load().sf_window_sync(self.handle, timeout_ms))

    def close(self):
        if self.handle:
            st = load().sf_window_destroy(self.handle)
            self.handle = None
            _check(st)

    def __del__(self):
        try:
            if self.handle:
                load().sf_window_destroy(self.handle)
        except Exception:
            pass


def sf_window_create(slots, h2d_stream, compute_stream, d2h_stream):
    """``slots``: list (one per slot) of lists of sf_tensor (device buffers)."""
    n_t = len(slots[0]) if slots else 0
    arrays = [tensor_array(s) for s in slots]
    ptrs = (ctypes.POINTER(sf_tensor) * max(1, len(slots)))()
    for i, a in enumerate(arrays):
        ptrs[i] = ctypes.cast(a, ctypes.POINTER(sf_tensor))
    h = ctypes.c_void_p()
    _check(load().sf_window_create(len(slots), ptrs, n_t, _stream(h2d_stream), _stream(compute_stream),
                                   _stream(d2h_stream), ctypes.byref(h)))
    return Window(h.value, (arrays, ptrs))


def host_layers(layers):
    """``layers``: list of lists of sf_tensor (pinned host buffers)."""
    arrays = [tensor_array(l) for l in layers]
    out = (sf_host_layer * max(1, len(layers)))()
    for i, (a, l) in enumerate(zip(arrays, layers)):
        out[i] = sf_host_layer(ctypes.cast(a, ctypes.POINTER(sf_tensor)), len(l))
    return out, arrays


def sf_slide_window_step(window, layers, order, hp, steps):
    """``layers`` from ``host_layers``; ``steps`` a ctypes int64 array (updated)."""
    hl, keep = layers
    n_layers = len(keep)
    order_arr = (ctypes.c_int32 * max(1, len(order)))(*order)
    _check(load().sf_slide_window_step(window.handle, hl, n_layers, order_arr, len(order), ctypes.byref(hp),
                                       steps))


# ----------------------------------------------------------------- (b') ----

class LspWindow:
    """Owning wrapper of an lsp_window handle; keeps its slot array alive."""

    def __init__(self, handle, keep):
        self.handle = handle
        self._keep = keep

    def sync(self, timeout_ms=0):
        _check(load().lsp_window_sync(self.handle, timeout_ms))

    def close(self):
        if self.handle:
            st = load().lsp_window_destroy(self.handle)
            self.handle = None
            _check(st)

    def __del__(self):
        try:
            if self.handle:
                load().lsp_window_destroy(self.handle)
        except Exception:
            pass


def lsp_window_create(slots, d, h2d_stream, compute_stream, d2h_stream):
    """``slots``: list of (S, m, v, dS, ws, ws_bytes) device buffers."""
    arr = (lsp_slot * max(1, len(slots)))()
    for i, (S, m, v, dS, ws, wsb) in enumerate(slots):
        arr[i] = lsp_slot(_addr(S), _addr(m), _addr(v), _addr(dS), _addr(ws), wsb)
    h = ctypes.c_void_p()
    _check(load().lsp_window_create(len(slots), arr, d, _stream(h2d_stream), _stream(compute_stream),
                                    _stream(d2h_stream), ctypes.byref(h)))
    return LspWindow(h.value, arr)


def lsp_window_create_host_update(slots, d, h2d_stream, compute_stream, d2h_stream, n_threads=0):
    """``slots``: list of (S, dS, S_host, dS_host, ws, ws_bytes): device S, dS, ws; pinned host staging."""
    arr = (lsp_host_slot * max(1, len(slots)))()
    for i, (S, dS, Sh, dSh, ws, wsb) in enumerate(slots):
        arr[i] = lsp_host_slot(_addr(S), _addr(dS), _addr(Sh), _addr(dSh), _addr(ws), wsb)
    h = ctypes.c_void_p()
    _check(load().lsp_window_create_host_update(len(slots), arr, d, int(n_threads), _stream(h2d_stream),
                                                _stream(compute_stream), _stream(d2h_stream), ctypes.byref(h)))
    return LspWindow(h.value, arr)


def lsp_window_timeline_start(window, capacity):
    _check(load().lsp_window_timeline_start(window.handle, int(capacity)))


def lsp_window_timeline_read(window, capacity):
    """Per recorded visit: [compress start, end, S copy start, end, host update end, dS copy start, end,
    apply start, end] in ms after the first point."""
    buf = (ctypes.c_float * max(1, capacity * 9))()
    n = ctypes.c_int(0)
    _check(load().lsp_window_timeline_read(window.handle, buf, int(capacity), ctypes.byref(n)))
    return [list(buf[v * 9:(v + 1) * 9]) for v in range(n.value)]


def lsp_layers(items):
    """``items``: list of dicts with P, Q, G, g_dtype, W, w_dtype, mirror, m, n, m_host, v_host."""
    arr = (lsp_layer * max(1, len(items)))()
    for i, it in enumerate(items):
        arr[i] = lsp_layer(it["P"].handle, it["Q"].handle, _addr(it["G"]), it["g_dtype"], _addr(it["W"]),
                           it["w_dtype"], _addr(it.get("mirror")), it["m"], it["n"], _addr(it["m_host"]),
                           _addr(it["v_host"]))
    return arr, items


def lsp_slide_window_step(window, layers, order, hp, steps):
    """``layers`` from ``lsp_layers``; ``steps`` a ctypes int64 array (updated)."""
    arr, items = layers
    order_arr = (ctypes.c_int32 * max(1, len(order)))(*order)
    _check(load().lsp_slide_window_step(window.handle, arr, len(items), order_arr, len(order), ctypes.byref(hp),
                                        steps))


def sf_sync_status(stream=None):
    _check(load().sf_sync_status(_stream(stream)))


def sf_last_error():
    return load().sf_last_error().decode()


def sf_version():
    return load().sf_version().decode()


def sf_test_device_wait_runs_out(limit_cycles, stream=None):
    _check(load().sf_test_device_wait_runs_out(limit_cycles, _stream(stream)))


def sf_test_fail_copy_after(n):
    load().sf_test_fail_copy_after(n)

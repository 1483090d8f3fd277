"""Benchmark of the per-layer update step on GB300.

Workload (the headline line): the LLaMA-2-7B-shaped full-parameter step,
32 decoder layers (hidden 4096, SwiGLU FFN 11008) plus the vocab-32000
embedding and LM head and the final norm, 6,738,415,616 params, seeded
synthetic bf16 gradients N(0, 1e-3) and fp32 master weights N(0, 0.02),
master/m/v all resident in HBM (108 GB with the bf16 gradient and weight
arrays).  One step = one fused multi-tensor AdamW launch per group in
sliding (backward) order: LM head, final norm, layers 31..0, embedding;
t advances per step.  Metric: params updated per second.

Also on the same line:
  e2e        the same step through the layer-sliding window with the fp32
             states kept resident in HBM: every step the gradients come
             from pinned host memory and the bf16 weights go back to it
             (2 + 2 bytes per param over the host link), copies inside the
             timed region.
  roofline   of the dominant kernel (the fused AdamW), from CUDA events
             around every launch in the timed region.
  gpu_launches  kernels one step enqueues (counted from a CUDA-graph
             capture of a step) times the timed steps.
  opt13      the OPT-1.3B-shaped stack (24 layers, 50,339,840 params each)
             resident in HBM, and its end-to-end form through the window
             with every array in pinned host memory (14 + 14 bytes per
             param over the link, 3 device slots).
  mistral_window  four Mistral-Large-123B-shaped layers (1.38 B params
             each) in pinned host memory streamed through 2 device slots,
             88 visits: link GB/s each way, overlap efficiency, and the
             update kernel's HBM fraction on one visit alone.
  lsp        the sparse-projector chain on the seven LLaMA-7B weight
             gradients (compress, compressed AdamW, decompress-apply into
             bf16 W; d = 512, 8 nonzeros per row), per-stage times, the
             chain replayed from CUDA graphs, the projector fit step, and
             the measured on-chip gather rates that bound the chain's
             kernels (shared memory, tensor memory, L2: gather_roof).
  lce        the fused linear cross-entropy on a Llama-3.1-8B output layer
             (8192 tokens, V 128256), tensor roofline against the burst
             bf16 figure (the sustained one when its clock record shows the
             power cap), with clocks.
  host_update  the same AdamW on the host cores (the pages' placement).
  cpu_baseline  the fp64 oracle on this machine's host cores, on a bounded
             sample of the same workload, with the CPU model, the cores the
             process may run on and numpy's BLAS threads.
  clocks     SM clocks and throttle reasons sampled during the timed region.

``--workload opt-1.3b`` or ``--workload mistral-window`` put one of the
other two workloads on the headline instead.  ``--impl reference`` times
the fp64 oracle instead (the only reference implementation of this path),
one bounded sample per step.

Multi-GPU (torchrun): every rank runs its own replica of the workload on
its own GPU; there is no collective on the data path.  ``value`` is the
params all ranks updated divided by the slowest rank's time.
"""

import argparse
import ctypes
import contextlib
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HP = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
ADAM_BYTES_PER_PARAM = 28        # 2 B grad + 3 x (4 B read + 4 B write) + 2 B bf16 weight
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0   # dense bf16, burst (no measured-peaks file on this machine)
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0   # the same under the power cap, seconds-long loop


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-lsp", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-lce", action="store_true")
    ap.add_argument("--layers", type=int, default=24, help="OPT-1.3B layers (24 = the full stack)")
    ap.add_argument("--workload", default="llama2-7b", choices=["llama2-7b", "opt-1.3b", "mistral-window"],
                    help="llama2-7b: the full LLaMA-2-7B step resident in HBM (headline); opt-1.3b: the 24-layer "
                         "OPT-1.3B stack; mistral-window: four Mistral-Large layers in pinned host memory through "
                         "2 device slots")
    ap.add_argument("--no-c5", action="store_true", help="leave out the Mistral-Large window sub-object")
    ap.add_argument("--profile-small", action="store_true",
                    help="1 layer, 1 warm-up + 1 timed step, no extras: a small case for ncu captures")
    ap.add_argument("--profile-lce", action="store_true",
                    help="only the fused linear cross-entropy on 2048 tokens of a LLaMA-2-7B output layer "
                         "(V 32000), 1 warm-up + 1 timed call: a small case for ncu captures")
    ap.add_argument("--profile-lsp", action="store_true",
                    help="only the projector chain on one 4096 x 4096 matrix, 1 warm-up + 1 timed rep (ncu case)")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers --

def dist_init(args):
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))   # this rank's GPU before its communicator
        dist.init_process_group(backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, units_per_step_per_rank, steps, slowest_ms):
    """Whole-job throughput: units all ranks processed over the slowest rank's time."""
    return world * units_per_step_per_rank * steps / (slowest_ms / 1e3)


def measured_peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBps", "hbm"):
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k]), "measured"
            for k, v in d.items():
                if "hbm" in k.lower() and isinstance(v, (int, float)):
                    return float(v), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def measured_peak_bf16(sustained=False):
    """Dense bf16 tensor peak in TFLOP/s, measured if the file has it, else the fallback.

    burst: a kernel timed alone; sustained: a kernel timed inside a long
    step, where the power cap holds the clocks down (the cross-entropy's ten
    16 ms calls in a row run with sw_power_cap active).
    """
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    keys = ("bf16_tflops_sustained", "bf16_TFLOPs_sustained") if sustained else ("bf16_tflops", "bf16_TFLOPs")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in keys:
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k]), "measured"
        except Exception:
            pass
    return (FALLBACK_BF16_TFLOPS_SUSTAINED if sustained else FALLBACK_BF16_TFLOPS), "fallback"


def kernel_traffic(kernel, units_per_launch=None):
    """dram bytes per launch from a committed ncu summary, if the kernel source is unchanged.

    The capture is of one smaller launch; the update's traffic grows in
    proportion to the params it updates, so with ``units_per_launch`` the
    captured bytes are scaled to a launch of that many params.
    """
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["source_sha"]:
        return None
    d = dict(d)
    if units_per_launch and d.get("unit_params_per_launch"):
        d["bytes_per_launch"] = d["bytes_per_launch"] * units_per_launch / d["unit_params_per_launch"]
        d["scaled_from_params"] = d["unit_params_per_launch"]
    return d


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""

    Q = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = bus_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            if self.bus_id and self.bus_id.lower() not in f[0].lower():
                continue
            self.rows.append(f)

    def summary(self):
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def bus_id_of_current_device():
    import torch
    try:
        pr = torch.cuda.get_device_properties(torch.cuda.current_device())
        return "%04x:%02x:%02x" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
    except Exception:
        return None


# ------------------------------------------------------------- CPU oracle --

def oracle_params_per_s(budget_s=12.0, chunk=1 << 21, max_steps=None):
    """fp64 oracle AdamW on chunks of an OPT-1.3B layer until the budget is spent."""
    import numpy as np
    import torch

    from layer_optimizer_gb300 import synth
    from oracle import adamw as oa
    th = synth.normal((chunk,), 0.02, 1).double().numpy()
    g = synth.normal((chunk,), 1e-3, 2, dtype=torch.bfloat16).float().double().numpy()
    st = oa.AdamWState(th)
    done, t0, t = 0, time.perf_counter(), 0
    while True:
        t += 1
        oa.adamw_step(st, g, t, **HP)
        done += chunk
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and t >= max_steps):
            break
    return done / el, done, el


def oracle_lsp_chain_rate(m=4096, n=4096, d=512, k=8):
    """fp64 oracle compress + compressed AdamW + decompress-apply on one LLaMA-7B q matrix (params/s)."""
    import numpy as np

    from layer_optimizer_gb300 import synth
    from oracle import adamw as oa
    from oracle import lsp as ol
    P = ol.Projector(*synth.projector(m, d, k, 1), d)
    Q = ol.Projector(*synth.projector(n, d, k, 2), d)
    rng = np.random.default_rng(3)
    G = rng.normal(0.0, 1e-3, size=(m, n))
    W = rng.normal(0.0, 0.02, size=(m, n))
    t0 = time.perf_counter()
    S, _ = ol.compress(P, Q, G)
    dS, *_ = oa.compressed_adamw_step(S, np.zeros((d, d)), np.zeros((d, d)), 1, HP["lr"], HP["beta1"],
                                      HP["beta2"], HP["eps"])
    D, _ = ol.decompress(P, Q, dS)
    ol.apply_fp32(W, D)
    el = time.perf_counter() - t0
    return {"params_per_s": m * n / el, "s": el,
            "sample": f"one {m} x {n} matrix, d {d}, k {k}: fp64 numpy (dense projector products)"}


def oracle_lce_rate(N=64, D=4096, V=128256):
    """fp64 oracle linear cross-entropy (loss, dH, dW) on a sample of tokens (tokens/s)."""
    import numpy as np

    from oracle.lce import lce
    rng = np.random.default_rng(4)
    H = rng.standard_normal((N, D), dtype=np.float32)
    W = rng.standard_normal((V, D), dtype=np.float32) * np.float32(0.02)
    y = rng.integers(0, V, size=N)
    t0 = time.perf_counter()
    lce(H, W, y)
    el = time.perf_counter() - t0
    return {"tokens_per_s": N / el, "s": el,
            "sample": f"{N} tokens of the same output layer (D {D}, V {V}): fp64 numpy, BLAS threads as installed"}


# ------------------------------------------------------------------ ours ---

def make_groups(groups, seed=0):
    """Device buffers for a list of tensor groups (one group = one launch)."""
    import torch

    from layer_optimizer_gb300 import synth
    out = []
    for li, grp in enumerate(groups):
        ts = []
        for ti, (_, n) in enumerate(grp):
            g = synth.fill_normal_(torch.empty(n, dtype=torch.bfloat16, device="cuda"), 1e-3,
                                   synth.sub_seed(seed, 1, li, ti))
            p = synth.fill_normal_(torch.empty(n, device="cuda"), 0.02, synth.sub_seed(seed, 2, li, ti))
            ts.append([g, p, torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda"),
                       torch.empty(n, dtype=torch.bfloat16, device="cuda")])
        out.append(ts)
    return out


def workload_groups(name, layers=24):
    from layer_optimizer_gb300 import synth
    if name == "llama2-7b":
        return synth.llama7_step_order()
    return [synth.OPT13_LAYER] * layers


def _cudart():
    """The CUDA runtime this process already loaded (torch and the library share it)."""
    for line in open("/proc/self/maps"):
        if "libcudart.so" in line:
            return ctypes.CDLL(line.split()[-1])
    return ctypes.CDLL("libcudart.so")


def kernels_per_call(fn, stream):
    """Kernel launches `fn()` enqueues on `stream`, counted from a CUDA-graph capture.

    The calls are captured (relaxed mode) into a graph that is never
    launched, so nothing runs and no state changes on the device.
    """
    rt = _cudart()
    rt.cudaStreamBeginCapture.argtypes = [ctypes.c_void_p, ctypes.c_int]
    rt.cudaStreamEndCapture.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
    rt.cudaGraphGetNodes.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)]
    rt.cudaGraphNodeGetType.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    rt.cudaGraphDestroy.argtypes = [ctypes.c_void_p]
    rt.cudaGetLastError.restype = ctypes.c_int
    sp = ctypes.c_void_p(stream.cuda_stream)
    if rt.cudaStreamBeginCapture(sp, 2) != 0:      # cudaStreamCaptureModeRelaxed
        rt.cudaGetLastError()                        # leave no error behind for the next launch
        return None
    graph = ctypes.c_void_p()
    try:
        fn()
    finally:
        rc = rt.cudaStreamEndCapture(sp, ctypes.byref(graph))
    if rc != 0 or not graph.value:
        rt.cudaGetLastError()
        return None
    n = ctypes.c_size_t(0)
    rt.cudaGraphGetNodes(graph, None, ctypes.byref(n))
    nodes = (ctypes.c_void_p * max(1, n.value))()
    rt.cudaGraphGetNodes(graph, nodes, ctypes.byref(n))
    kernels = 0
    for k in range(n.value):
        t = ctypes.c_int(-1)
        rt.cudaGraphNodeGetType(nodes[k], ctypes.byref(t))
        kernels += t.value == 0                      # cudaGraphNodeTypeKernel
    rt.cudaGraphDestroy(graph)
    return kernels


def host_mem_available():
    """Bytes of host memory the kernel reports as available (MemAvailable), or None."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def pinned_leg_fits(bytes_per_rank, local_ranks, available, headroom=1.3):
    """Whether every rank on this node can pin `bytes_per_rank` of host memory at once.

    `available` is MemAvailable read before any rank pinned anything; the
    ranks of one node share it.  Unknown memory counts as not enough.
    """
    if available is None:
        return False
    return bytes_per_rank * local_ranks * headroom <= available


def release_pinned():
    """Hand torch's cached pinned host blocks back to the system."""
    import torch
    f = getattr(torch._C, "_host_emptyCache", None)
    if f is not None:
        f()


def cpu_context():
    """The host the oracle runs on: CPU model, usable cores, numpy's BLAS threads."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            model = None
    blas = {k: os.environ[k] for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
            if k in os.environ}
    return {"cpu_model": model or "unknown", "affinity_cores": len(os.sched_getaffinity(0)),
            "os_cpu_count": os.cpu_count(),
            "blas_threads": blas or "library default (all usable cores); the elementwise oracle runs single-threaded"}


def run_resident(args, world, groups, keep=False):
    import torch

    from layer_optimizer_gb300 import native, synth
    layers = make_groups(groups)
    params_per_step = sum(synth.layer_numel(g) for g in groups)
    hp = native.hparams(**HP)
    descs = [[native.make_tensor(*t) for t in L] for L in layers]
    arrs = [native.tensor_array(d) for d in descs]
    lib = native.load()
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    step = [0]
    n_groups = len(groups)

    def one_step(evs=None, t=None, sp=sptr):
        if t is None:
            step[0] += 1
            t = step[0]
        for li, a in enumerate(arrs):
            if evs is not None:
                evs[li][0].record(stream)
            st = lib.sf_adamw_layer_step(a, len(descs[li]), ctypes.byref(hp), t, sp)
            if st != 0:
                raise native.SfError(st, native.sf_last_error())
            if evs is not None:
                evs[li][1].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()          # graph capture needs a stream other than the legacy default one
    per_step = kernels_per_call(lambda: one_step(t=step[0] + 1, sp=side.cuda_stream), side)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_groups)]
           for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clk = Clocks(bus_id_of_current_device())
    with clk:
        t0.record(stream)
        for k in range(args.steps):
            one_step(evs[k])
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    total_ms = t0.elapsed_time(t1)
    launch_ms = [a.elapsed_time(b) for row in evs for (a, b) in row]
    group_params = [synth.layer_numel(g) for g in groups] * args.steps
    out = dict(total_ms=total_ms, launch_ms=launch_ms, params_per_step=params_per_step, group_params=group_params,
               launches=per_step * args.steps if per_step is not None else None, kernels_per_step=per_step,
               clocks=clk.summary(), steps_done=step[0])
    if keep:
        out["layers"] = layers
    else:
        del layers
        torch.cuda.empty_cache()
    return out


def resident_summary(res, args, world):
    """Value, step time and roofline of a resident run (whole job over the slowest rank)."""
    total_ms = max_over_ranks(res["total_ms"], world)
    lm = res["launch_ms"]
    peak, kind = measured_peak_hbm()
    achieved = ADAM_BYTES_PER_PARAM * sum(res["group_params"]) / (sum(lm) / 1e3) / 1e9
    traffic = kernel_traffic("adamw_bulk_kernel", sum(res["group_params"]) / len(res["group_params"]))
    return {
        "value": job_value(world, res["params_per_step"], args.steps, total_ms),
        "ms_per_step": total_ms / args.steps,
        "roofline": {"bound": "hbm", "kernel": "adamw_bulk_kernel", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{kind} ({'of measured' if kind == 'measured' else 'of fallback'})",
                     "bytes_per_launch": ADAM_BYTES_PER_PARAM * sum(res["group_params"]) / len(res["group_params"]),
                     "avg_launch_ms": sum(lm) / len(lm),
                     "traffic": traffic["bytes_per_launch"] if traffic else None},
    }


def run_e2e_states_resident(args, world, groups, layers, start_step):
    """The resident step through the window: gradients in, bf16 weights out, fp32 states in HBM.

    Each group's gradient and weight arrays are flat pinned host buffers
    (the gradient holds the same bits as the resident run's); master, m and
    v are the resident run's device arrays, which the window updates in
    place.  Three device slots hold one group's gradient and weight each.
    """
    import torch

    from layer_optimizer_gb300 import native, synth
    bf16 = torch.bfloat16
    host, keep = [], []
    for gi, grp in enumerate(groups):
        n = synth.layer_numel(grp)
        hg = torch.empty(n, dtype=bf16, pin_memory=True)
        hw = torch.empty(n, dtype=bf16, pin_memory=True)
        keep += [hg, hw]
        off, ts = 0, []
        for ti, (_, c) in enumerate(grp):
            dg = layers[gi][ti]
            hg[off:off + c].copy_(dg[0])
            ts.append([hg[off:off + c], dg[1], dg[2], dg[3], hw[off:off + c]])
            off += c
        host.append(ts)
    torch.cuda.synchronize()
    # slot tensor i sits at its offset in the largest group; its capacity is
    # the largest tensor i of any group (a one-tensor group such as the LM
    # head overlaps the larger group's later tensors, which it never uses)
    n_t = max(len(g) for g in groups)
    big = max(groups, key=synth.layer_numel)
    offs = [sum(c for _, c in big[:i]) for i in range(len(big))]
    offs += [offs[-1]] * (n_t - len(offs))
    caps = [max(g[i][1] for g in groups if len(g) > i) for i in range(n_t)]
    slot_elems = max(o + c for o, c in zip(offs, caps))
    n_slots = 3
    slot_bufs = [(torch.empty(slot_elems, dtype=bf16, device="cuda"), torch.empty(slot_elems, dtype=bf16, device="cuda"))
                 for _ in range(n_slots)]
    slots = [[native.make_tensor(fg[o:o + c], None, None, None, fw[o:o + c], numel=c) for o, c in zip(offs, caps)]
             for fg, fw in slot_bufs]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.sf_window_create(slots, *streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L] for L in host])
    order = list(range(len(groups)))
    steps = (ctypes.c_int64 * len(groups))(*([start_step] * len(groups)))
    hp = native.hparams(**HP)
    native.sf_slide_window_step(win, hl, order, hp, steps)
    win.sync()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        native.sf_slide_window_step(win, hl, order, hp, steps)
    win.sync()
    wall = time.perf_counter() - t0
    barrier(world)
    params = sum(synth.layer_numel(g) for g in groups)
    win.close()
    del host, keep, slots, slot_bufs
    release_pinned()
    torch.cuda.empty_cache()
    return dict(wall_s=wall, params_per_step=params, h2d=2 * params, d2h=2 * params)


def link_probe(nbytes=2 << 30, reps=5):
    """Raw host<->device copy bandwidth with pinned buffers: each direction alone, then both at once."""
    import torch
    h_a = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_b = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d_b = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    def h2d():
        with torch.cuda.stream(s1):
            d_a.copy_(h_a, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_b.copy_(d_b, non_blocking=True)

    def both():
        h2d()
        d2h()
    h2d(); d2h(); torch.cuda.synchronize()
    t_h2d, t_d2h, t_both = timed(h2d), timed(d2h), timed(both)
    out = {"bytes": nbytes, "h2d_GBps": nbytes / t_h2d / 1e9, "d2h_GBps": nbytes / t_d2h / 1e9,
           "bidir_each_GBps": nbytes / t_both / 1e9}
    del h_a, h_b, d_a, d_b
    return out


def run_e2e(args, world):
    """Same step through the window engine with the layers in pinned host memory."""
    import torch

    from layer_optimizer_gb300 import native, synth
    n_layers = args.layers
    # each layer's arrays flat in pinned host memory (grad, master, m, v,
    # weight: one buffer each, the tensors views into it), as flattened
    # optimizer states are kept; the window then moves each array of a
    # layer as one copy
    sizes = [n for _, n in synth.OPT13_LAYER]
    per_layer = sum(sizes)
    dtypes = (torch.bfloat16, torch.float32, torch.float32, torch.float32, torch.bfloat16)

    def views(flat):
        out, o = [], 0
        for n in sizes:
            out.append([f[o:o + n] for f in flat])
            o += n
        return out
    host_flat, host = [], []
    for li in range(n_layers):
        flat = [torch.zeros(per_layer, dtype=dt, pin_memory=True) for dt in dtypes]
        ts = views(flat)
        for ti, n in enumerate(sizes):
            ts[ti][0].copy_(synth.fill_normal_(torch.empty(n, dtype=torch.bfloat16, device="cuda"), 1e-3,
                                               synth.sub_seed(3, li, ti)))
            ts[ti][1].copy_(synth.fill_normal_(torch.empty(n, device="cuda"), 0.02, synth.sub_seed(4, li, ti)))
        host_flat.append(flat)
        host.append(ts)
    # three device slots: a layer's update and write-back, the next layer's
    # copy in and a third layer's copy in can all be in flight (0.8 GB each)
    n_slots = 3
    slot_flat = [[torch.empty(per_layer, dtype=dt, device="cuda") for dt in dtypes] for _ in range(n_slots)]
    slots = [views(f) for f in slot_flat]
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.sf_window_create([[native.make_tensor(*t) for t in s] for s in slots], *streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L] for L in host])
    steps = (ctypes.c_int64 * n_layers)()
    hp = native.hparams(**HP)
    order = list(range(n_layers))
    for _ in range(max(1, args.warmup)):
        native.sf_slide_window_step(win, hl, order, hp, steps)
    win.sync()
    # the same pinned buffers copied with plain bidirectional copies (no
    # engine, no kernel, no events): the link rate these buffers allow
    torch.cuda.synchronize()
    tr = time.perf_counter()
    for li, F in enumerate(host_flat):
        with torch.cuda.stream(streams[0]):
            for k in range(4):
                slot_flat[li % n_slots][k].copy_(F[k], non_blocking=True)
        with torch.cuda.stream(streams[2]):
            for k in (1, 2, 3, 4):
                F[k].copy_(slot_flat[(li + 1) % n_slots][k], non_blocking=True)
    torch.cuda.synchronize()
    raw_s = time.perf_counter() - tr
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        native.sf_slide_window_step(win, hl, order, hp, steps)
    win.sync()
    wall = time.perf_counter() - t0
    barrier(world)
    params = n_layers * synth.layer_numel(synth.OPT13_LAYER)
    win.close()
    del host, slots, host_flat, slot_flat
    torch.cuda.empty_cache()
    return dict(wall_s=wall, params_per_step=params, h2d=14 * params, d2h=14 * params,
                raw_copy_GBps_each_way=14 * params / raw_s / 1e9)


def run_lsp(args, matrices=None):
    """Compress -> compressed AdamW -> decompress-apply on the LLaMA-7B matrices."""
    import torch

    from layer_optimizer_gb300 import native, synth
    d, k = 512, 8
    hp = native.hparams(**HP)
    mats = []
    for mi, (name, m, n) in enumerate(matrices or synth.LLAMA7_LSP_MATRICES):
        Pi, Pv = synth.projector(m, d, k, synth.sub_seed(7, mi, 0))
        Qi, Qv = synth.projector(n, d, k, synth.sub_seed(7, mi, 1))
        P = native.lsp_projector_create(m, d, k, torch.from_numpy(Pi).cuda(), torch.from_numpy(Pv).cuda())
        Q = native.lsp_projector_create(n, d, k, torch.from_numpy(Qi).cuda(), torch.from_numpy(Qv).cuda())
        G = synth.fill_normal_(torch.empty(m, n, device="cuda"), 1e-3, synth.sub_seed(8, mi))
        W = synth.fill_normal_(torch.empty(m, n, dtype=torch.bfloat16, device="cuda"), 0.02, synth.sub_seed(9, mi))
        st = [torch.zeros(d, d, device="cuda") for _ in range(4)]  # S, m, v, dS
        wsb = native.lsp_workspace_bytes(m, n, d)
        ws = torch.empty(max(16, wsb), dtype=torch.uint8, device="cuda")
        mats.append((name, m, n, P, Q, G, W, st, ws, wsb))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    reps = 1 if args.profile_lsp else max(3, args.steps // 2)
    times = {"compress": [], "adamw_c": [], "decompress": []}
    per = []
    for it in range(args.warmup + reps):
        row = []
        for (name, m, n, P, Q, G, W, (S, mm, vv, dS), ws, wsb) in mats:
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(stream)
            native.lsp_compress(P, Q, G, native.SF_FP32, m, n, S, ws, wsb, stream)
            e[1].record(stream)
            native.lsp_adamw_compressed(S, mm, vv, dS, d * d, hp, it + 1, stream)
            e[2].record(stream)
            native.lsp_decompress_apply(P, Q, dS, W, native.SF_BF16, None, m, n, ws, wsb, stream)
            e[3].record(stream)
            row.append((m, n, e))
        torch.cuda.synchronize()
        if it >= args.warmup:
            for m, n, e in row:
                per.append((m, n, e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3])))
    # the layer's compress in one call (first stages of all matrices in one
    # launch, second stages in another), eager, same inputs
    layer_ms = None
    try:
        ms_, ns_ = [x[1] for x in mats], [x[2] for x in mats]
        wlb = native.lsp_compress_layer_workspace_bytes(ms_, ns_, d)
        wl = torch.empty(wlb, dtype=torch.uint8, device="cuda")
        Ps_, Qs_, Gs_ = [x[3] for x in mats], [x[4] for x in mats], [x[5] for x in mats]
        Ss_ = [x[7][0] for x in mats]
        for _ in range(args.warmup):
            native.lsp_compress_layer(Ps_, Qs_, Gs_, [native.SF_FP32] * len(mats), ms_, ns_, Ss_, wl, wlb, stream)
        torch.cuda.synchronize()
        lt = []
        for _ in range(reps):
            la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            la.record(stream)
            native.lsp_compress_layer(Ps_, Qs_, Gs_, [native.SF_FP32] * len(mats), ms_, ns_, Ss_, wl, wlb, stream)
            lb.record(stream)
            torch.cuda.synchronize()
            lt.append(la.elapsed_time(lb))
        layer_ms = sorted(lt)[len(lt) // 2]
        del wl
    except Exception as ex:  # recorded on the line, the per-call numbers still stand
        layer_ms = f"layer compress failed: {str(ex)[:120]}"
    # the same chain for all matrices captured once in a CUDA graph and
    # replayed: no host gaps between the launches
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            cs = torch.cuda.current_stream()
            for (name, m, n, P, Q, G, W, (S, mm, vv, dS), ws, wsb) in mats:
                native.lsp_compress(P, Q, G, native.SF_FP32, m, n, S, ws, wsb, cs)
                native.lsp_adamw_compressed(S, mm, vv, dS, d * d, hp, args.warmup + reps + 1, cs)
                native.lsp_decompress_apply(P, Q, dS, W, native.SF_BF16, None, m, n, ws, wsb, cs)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record(stream)
        for _ in range(reps):
            g.replay()
        gb.record(stream)
        torch.cuda.synchronize()
        graph_ms = ga.elapsed_time(gb) / reps
        del g
    except Exception as ex:  # recorded on the line, eager numbers still stand
        graph_ms = f"graph capture failed: {str(ex)[:120]}"
    # the matrices are independent: one stream per matrix chain inside one
    # graph lets the small kernels of one chain overlap the large ones of another
    graph_ms_streams = None
    try:
        g2 = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        side = [torch.cuda.Stream() for _ in mats]
        with torch.cuda.graph(g2, stream=cap):
            root = torch.cuda.current_stream()
            for st_, (name, m, n, P, Q, G, W, (S, mm, vv, dS), ws, wsb) in zip(side, mats):
                st_.wait_stream(root)
                native.lsp_compress(P, Q, G, native.SF_FP32, m, n, S, ws, wsb, st_)
                native.lsp_adamw_compressed(S, mm, vv, dS, d * d, hp, args.warmup + reps + 2, st_)
                native.lsp_decompress_apply(P, Q, dS, W, native.SF_BF16, None, m, n, ws, wsb, st_)
            for st_ in side:
                root.wait_stream(st_)
        torch.cuda.synchronize()
        g2.replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record(stream)
        for _ in range(reps):
            g2.replay()
        gb.record(stream)
        torch.cuda.synchronize()
        graph_ms_streams = ga.elapsed_time(gb) / reps
        del g2
    except Exception as ex:
        graph_ms_streams = f"multi-stream graph failed: {str(ex)[:120]}"
    # the same chain with the compressed moments in pinned host memory,
    # through the layer-wise window (2 device slots, 3 streams)
    host_ms = None
    try:
        items = []
        for (name, m, n, P, Q, G, W, (S, mm, vv, dS), ws, wsb) in mats:
            items.append(dict(P=P, Q=Q, G=G, g_dtype=native.SF_FP32, W=W, w_dtype=native.SF_BF16, m=m, n=n,
                              m_host=torch.zeros(d, d).pin_memory(), v_host=torch.zeros(d, d).pin_memory()))
        wsb_max = max(x[9] for x in mats)
        slots = [tuple(torch.zeros(d, d, device="cuda") for _ in range(4)) +
                 (torch.empty(wsb_max, dtype=torch.uint8, device="cuda"), wsb_max) for _ in range(2)]
        wstreams = [torch.cuda.Stream() for _ in range(3)]
        lw = native.lsp_window_create(slots, d, *wstreams)
        lay = native.lsp_layers(items)
        lsteps = (ctypes.c_int64 * len(items))()
        order = list(range(len(items)))
        for _ in range(args.warmup):
            native.lsp_slide_window_step(lw, lay, order, hp, lsteps)
        lw.sync()
        t0 = time.perf_counter()
        for _ in range(reps):
            native.lsp_slide_window_step(lw, lay, order, hp, lsteps)
        lw.sync()
        host_ms = (time.perf_counter() - t0) / reps * 1e3
        lw.close()
        del slots
    except Exception as ex:
        host_ms = f"host-moment window failed: {str(ex)[:120]}"
        items = None
    # LSP-Offload's own placement: S to the host, the compressed AdamW on the
    # host cores, dS back (3 slots: the host round trip of one matrix
    # overlaps the next ones' compress), then a timeline of one pass
    host_upd = None
    try:
        if items is None:
            raise RuntimeError("no layer list")
        for it in items:
            it["m_host"].zero_()
            it["v_host"].zero_()
        wsb_max = max(x[9] for x in mats)
        hslots = [(torch.zeros(d, d, device="cuda"), torch.zeros(d, d, device="cuda"), torch.zeros(d, d).pin_memory(),
                   torch.zeros(d, d).pin_memory(), torch.empty(wsb_max, dtype=torch.uint8, device="cuda"), wsb_max)
                  for _ in range(3)]
        wstreams = [torch.cuda.Stream() for _ in range(3)]
        hw = native.lsp_window_create_host_update(hslots, d, *wstreams)
        lay = native.lsp_layers(items)
        lsteps = (ctypes.c_int64 * len(items))()
        order = list(range(len(items)))
        for _ in range(args.warmup):
            native.lsp_slide_window_step(hw, lay, order, hp, lsteps)
        hw.sync()
        t0 = time.perf_counter()
        for _ in range(reps):
            native.lsp_slide_window_step(hw, lay, order, hp, lsteps)
        hw.sync()
        hu_ms = (time.perf_counter() - t0) / reps * 1e3
        native.lsp_window_timeline_start(hw, len(items))
        native.lsp_slide_window_step(hw, lay, order, hp, lsteps)
        tl = native.lsp_window_timeline_read(hw, len(items))
        hw.close()
        wall = max(v[8] for v in tl) - min(v[0] for v in tl)
        gpu = sum((v[1] - v[0]) + (v[8] - v[7]) for v in tl)
        link = sum((v[3] - v[2]) + (v[6] - v[5]) for v in tl)
        host = sum(v[4] - v[3] for v in tl)
        host_upd = {"ms_per_chain_all7": hu_ms, "params_per_s": sum(m * n for (_, m, n, *_r) in mats) / (hu_ms / 1e3),
                    "link_bytes_each_way_per_chain": 4 * d * d * len(items),
                    "host_threads": min(8, len(os.sched_getaffinity(0))),
                    "timeline_one_pass_ms": {"wall": wall, "gpu_compress_and_apply": gpu, "link_copies": link,
                                             "host_updates": host,
                                             "overlap_efficiency": max(gpu, link, host) / wall if wall > 0 else None},
                    "timeline_visits": [[round(x, 4) for x in v] for v in tl],
                    "timeline_points": "compress start, end; S to host start, end; host update end; dS to device "
                                       "start, end; decompress-apply start, end (ms)"}
        del hslots
    except Exception as ex:
        host_upd = {"error": f"host-update window failed: {str(ex)[:160]}"}
    # projector fit step (gradient descent on the stored values of P and Q
    # for the reconstruction error of G), once per matrix, after everything
    # above so that the changed values touch no other measurement
    fit_ms = None
    try:
        wsf = max(native.lsp_fit_workspace_bytes(m, n, d, native.SF_FP32) for (_, m, n, *_r) in mats)
        wsf_t = torch.empty(wsf, dtype=torch.uint8, device="cuda")
        loss = torch.empty(len(mats), dtype=torch.float64, device="cuda")

        def fit_all():
            for i, (name, m, n, P, Q, G, W, st4, ws, wsb) in enumerate(mats):
                native.lsp_projector_fit_step(P, Q, G, native.SF_FP32, m, n, 1e-9, loss[i:i + 1], None, None,
                                              wsf_t, wsf, stream)
        for _ in range(args.warmup):
            fit_all()
        torch.cuda.synchronize()
        fa, fb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fa.record(stream)
        for _ in range(reps):
            fit_all()
        fb.record(stream)
        torch.cuda.synchronize()
        fit_ms = fa.elapsed_time(fb) / reps
        del wsf_t
    except Exception as ex:
        fit_ms = f"fit step failed: {str(ex)[:120]}"
    # the second roof of these kernels: gathered multiply-adds per second
    # with every operand in shared memory (the gather kernels' inner loop alone)
    gather_rate = None
    try:
        nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        sink = torch.empty(nsm * 512, device="cuda")
        native.sf_bench_gather_rate(nsm, 1024, sink, stream)
        torch.cuda.synchronize()
        ra, rb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        iters = 1 << 15
        ra.record(stream)
        native.sf_bench_gather_rate(nsm, iters, sink, stream)
        rb.record(stream)
        torch.cuda.synchronize()
        gather_rate = nsm * 512 * iters * 8 / (ra.elapsed_time(rb) / 1e3)
    except Exception as ex:
        gather_rate = f"gather-rate probe failed: {str(ex)[:120]}"
    # the other on-chip source: tensor memory (tcgen05.ld of 1, 2 or 4
    # columns per lane at columns chosen per load, entries from shared
    # memory), and row gathers straight from L2 (a 48 MB buffer)
    other_roofs = {}
    try:
        def timed_call(fn):
            fn()
            torch.cuda.synchronize()
            ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ea.record(stream)
            fn()
            eb.record(stream)
            torch.cuda.synchronize()
            return ea.elapsed_time(eb) / 1e3
        tm = {}
        for x in (1, 2, 4):
            it = (1 << 14) // x
            t = timed_call(lambda: native.sf_bench_tmem_rate(nsm, it, x, 1, sink, stream))
            tm[f"x{x}_macs_per_s"] = nsm * 512 * it * 8 * x / t
        other_roofs["tmem"] = dict(tm, probe="sf_bench_tmem_rate: 16 warps per SM, 8 tcgen05.ld.32x32b.xN per "
                                             "wait, column and multiplier per load from a shared-memory entry")
        rows = 48 * 2048
        buf = torch.rand(rows, 128, device="cuda")
        sk = torch.empty(nsm * 2 * 256, device="cuda")
        t = timed_call(lambda: native.sf_bench_l2_gather_rate(nsm * 2, 256, buf, rows, sk, stream))
        l2_bytes = nsm * 2 * 8 * 256 * 16 * 512
        other_roofs["l2_rows"] = {"GBps": l2_bytes / t / 1e9, "macs_per_s_fp32": l2_bytes / 4 / t,
                                  "probe": "sf_bench_l2_gather_rate: 512-byte rows of a 48 MB buffer, 16 loads in "
                                           "flight per lane, 2 CTAs of 8 warps per SM"}
        del buf, sk
    except Exception as ex:
        other_roofs = {"error": f"tmem / L2 probes failed: {str(ex)[:120]}"}
    n_params = sum(m * n for (_, m, n, *_r) in mats)
    comp_t = sum(p[2] for p in per) / reps
    ad_t = sum(p[3] for p in per) / reps
    dec_t = sum(p[4] for p in per) / reps
    comp_bytes = sum(m * n * 4 + d * d * 4 + (m + n) * k * 8 for (_, m, n, *_r) in mats)
    dec_bytes = sum(m * n * 4 + d * d * 4 + (m + n) * k * 8 for (_, m, n, *_r) in mats)
    peak, kind = measured_peak_hbm()
    out = {
        "workload": "LLaMA-7B q,k,v,o 4096x4096, gate/up 11008x4096, down 4096x11008; G fp32, W bf16; d=512, k=8",
        "params_updated_per_s": n_params / ((comp_t + ad_t + dec_t) / 1e3),
        "ms_per_chain_all7": comp_t + ad_t + dec_t,
        "compress": {"ms": comp_t, "GBps": comp_bytes / comp_t / 1e6, "frac": comp_bytes / comp_t / 1e6 / peak},
        "compress_layer": ({"ms": layer_ms, "GBps": comp_bytes / layer_ms / 1e6,
                            "frac": comp_bytes / layer_ms / 1e6 / peak,
                            "call": "lsp_compress_layer: the seven matrices in one call (two launches)"}
                           if isinstance(layer_ms, float) else layer_ms),
        "adamw_compressed": {"ms": ad_t},
        "decompress_apply": {"ms": dec_t, "GBps": dec_bytes / dec_t / 1e6, "frac": dec_bytes / dec_t / 1e6 / peak},
        "peak_GBps": peak, "peak_kind": kind,
        "ms_per_chain_all7_graph": graph_ms,
    }
    all_bytes = comp_bytes + dec_bytes + 24 * d * d * len(mats)
    if isinstance(graph_ms, float):
        out["params_updated_per_s_graph"] = n_params / (graph_ms / 1e3)
        out["chain_GBps_graph"] = all_bytes / graph_ms / 1e6
        out["chain_frac_graph"] = all_bytes / graph_ms / 1e6 / peak
    out["fit_step"] = {"ms_all7": fit_ms}
    if isinstance(fit_ms, float):
        g_bytes = sum(m * n * 4 for (_, m, n, *_r) in mats)
        out["fit_step"].update({"G_GBps": g_bytes / fit_ms / 1e6, "frac": g_bytes / fit_ms / 1e6 / peak,
                                "bytes": "G read once (m n 4 B per matrix) is the algorithmic minimum"})
    if isinstance(gather_rate, float):
        # compress: m n k (stage 1 over G) + n d k (stage 2); decompress:
        # d n k (V = dS Q^T) + m n k (apply); fp32 G at k = 8 is 2 MAC per byte
        comp_macs = sum(m * n * k + n * d * k for (_, m, n, *_r) in mats)
        dec_macs = sum(d * n * k + m * n * k for (_, m, n, *_r) in mats)
        out["gather_roof"] = {
            "macs_per_s": gather_rate,
            "as_hbm_fraction": gather_rate / (k / 4) / (peak * 1e9),
            "compress_frac": comp_macs / (comp_t / 1e3) / gather_rate,
            "decompress_frac": dec_macs / (dec_t / 1e3) / gather_rate,
            "probe": "sf_bench_gather_rate: 16 warps per SM, 2 entries + 2 float4 tile loads + 8 FMA per step"}
    else:
        out["gather_roof"] = {"error": gather_rate}
    out["gather_roof"].update(other_roofs)
    out["ms_per_chain_all7_graph_streams"] = graph_ms_streams
    out["ms_per_chain_all7_host_moments_window"] = host_ms
    out["host_update_window"] = host_upd
    if isinstance(host_ms, float):
        out["params_updated_per_s_host_moments_window"] = n_params / (host_ms / 1e3)
    if isinstance(graph_ms_streams, float):
        out["params_updated_per_s_graph_streams"] = n_params / (graph_ms_streams / 1e3)
        out["chain_frac_graph_streams"] = all_bytes / graph_ms_streams / 1e6 / peak
    for x in mats:
        x[3].close()
        x[4].close()
    del mats
    torch.cuda.empty_cache()
    return out


def run_lce(args, N=8192, D=4096, V=128256, chunk=4608):
    """Fused linear cross-entropy (loss, dH, dW) on a Llama-3.1-8B output layer.

    Chunks of 4608 tokens = 18 tiles of 256 rows (one per CTA pair): the dH
    product's 18 x 16 tiles take 3.8 of the 4 waves of 76 CTA pairs, the
    3584-token remainder's 14 x 16 tiles 2.95 of 3.
    """
    import torch

    from layer_optimizer_gb300 import native, synth
    H = synth.fill_normal_(torch.empty(N, D, dtype=torch.bfloat16, device="cuda"), 1.0, synth.sub_seed(21, 0))
    W = synth.fill_normal_(torch.empty(V, D, dtype=torch.bfloat16, device="cuda"), 0.02, synth.sub_seed(21, 1))
    g = torch.Generator(device="cuda")
    g.manual_seed(synth.sub_seed(21, 2))
    y = torch.randint(0, V, (N,), generator=g, device="cuda", dtype=torch.int32)
    wsb = native.lce_workspace_bytes(N, D, V, chunk)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    loss = torch.empty(1, dtype=torch.float64, device="cuda")
    dH = torch.empty(N, D, device="cuda")
    dW = torch.empty(V, D, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        native.lce_forward_backward(H, W, y, N, D, V, chunk, -100, loss, dH, dW, ws, wsb, stream)
    reps = 1 if args.profile_lce else max(5, args.steps // 2)
    for _ in range(1 if args.profile_lce else args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = Clocks(bus_id_of_current_device())
    with (contextlib.nullcontext() if args.profile_lce else clk):
        e0.record(stream)
        for _ in range(reps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    flops = 6.0 * N * V * D
    # the calls are a burst of well under a second: the burst figure is the
    # denominator unless this leg's own clock record shows the power cap
    clocks = clk.summary()
    capped = "sw_power_cap" in clocks.get("reasons", [])
    peak, kind = measured_peak_bf16(sustained=capped)
    burst, _ = measured_peak_bf16()
    sustained, _ = measured_peak_bf16(sustained=True)
    out = {"workload": f"Llama-3.1-8B output layer: {N} tokens, D {D}, V {V}, chunks of {chunk}; bf16 H and W, "
                       "fp32 dH and dW",
           "ms": ms, "tokens_per_s": N / (ms / 1e3),
           "roofline": {"bound": "tensor", "achieved": flops / ms / 1e9, "peak": peak, "unit": "TFLOP/s",
                        "frac": flops / ms / 1e9 / peak,
                        "peak_kind": f"{kind} {'sustained (power cap seen)' if capped else 'burst'} (of {kind})",
                        "frac_of_sustained_peak": flops / ms / 1e9 / sustained, "flops_per_call": flops,
                        "timed_region_ms": ms * reps},
           "logits_bytes_full": N * V * 4, "workspace_bytes": wsb, "loss": float(loss.item()), "calls": reps,
           "clocks": clocks}
    del H, W, dH, dW, ws
    torch.cuda.empty_cache()
    return out


def host_update_rate(steps=3):
    """The same AdamW step on all host cores (sf_adamw_host_step), one OPT-1.3B layer in host memory."""
    import torch

    from layer_optimizer_gb300 import native, synth
    layer = []
    for ti, (_, n) in enumerate(synth.OPT13_LAYER):
        layer.append([synth.normal((n,), 1e-3, synth.sub_seed(11, ti), dtype=torch.bfloat16),
                      synth.normal((n,), 0.02, synth.sub_seed(12, ti)), torch.zeros(n), torch.zeros(n),
                      torch.empty(n, dtype=torch.bfloat16)])
    ts = [native.make_tensor(*t) for t in layer]
    hp = native.hparams(**HP)
    threads = len(os.sched_getaffinity(0))
    native.sf_adamw_host_step(ts, hp, 1, threads)
    t0 = time.perf_counter()
    for k in range(steps):
        native.sf_adamw_host_step(ts, hp, k + 2, threads)
    el = (time.perf_counter() - t0) / steps
    n = synth.layer_numel(synth.OPT13_LAYER)
    return {"params_per_s": n / el, "GBps": ADAM_BYTES_PER_PARAM * n / el / 1e9, "threads": threads,
            "sample": f"one OPT-1.3B layer ({n} params) in host memory, {steps} steps",
            "note": "SlideFormer's own placement of the update (host cores), same arithmetic and bits as the GPU"}


def run_mistral_window(args, world):
    """Four Mistral-Large layers in pinned host memory streamed through 2 device slots, 88 visits."""
    import torch

    from layer_optimizer_gb300 import native, synth
    layer = synth.MISTRAL_LAYER
    n_phys, n_visits = 4, 88
    caps = [n for _, n in layer]
    chunk = 1 << 28
    tmp = torch.empty(chunk, device="cuda")
    tmpb = torch.empty(chunk, dtype=torch.bfloat16, device="cuda")
    zero = torch.zeros(chunk, device="cuda")

    def fill_pinned(t, std, seed):
        flat = t.view(-1)
        for ci, s0 in enumerate(range(0, flat.numel(), chunk)):
            e = min(flat.numel(), s0 + chunk)
            if std is None:
                flat[s0:e].copy_(zero[:e - s0])
            elif t.dtype == torch.float32:
                synth.fill_normal_(tmp[:e - s0], std, synth.sub_seed(seed, ci))
                flat[s0:e].copy_(tmp[:e - s0])
            else:
                synth.fill_normal_(tmpb[:e - s0], std, synth.sub_seed(seed, ci))
                flat[s0:e].copy_(tmpb[:e - s0])
        torch.cuda.synchronize()
        return t

    t_alloc = time.perf_counter()
    host = []
    for li in range(n_phys):
        ts = []
        for ti, n in enumerate(caps):
            g = fill_pinned(torch.empty(n, dtype=torch.bfloat16, pin_memory=True), 1e-3, synth.sub_seed(5, li, ti, 0))
            p = fill_pinned(torch.empty(n, pin_memory=True), 0.02, synth.sub_seed(5, li, ti, 1))
            m = fill_pinned(torch.empty(n, pin_memory=True), None, 0)
            v = fill_pinned(torch.empty(n, pin_memory=True), None, 0)
            w = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
            ts.append([g, p, m, v, w])
        host.append(ts)
    del tmp, tmpb, zero
    slots = [[[torch.empty(c, dtype=torch.bfloat16, device="cuda"), torch.empty(c, device="cuda"),
               torch.empty(c, device="cuda"), torch.empty(c, device="cuda"),
               torch.empty(c, dtype=torch.bfloat16, device="cuda")] for c in caps] for _ in range(2)]
    setup_s = time.perf_counter() - t_alloc
    streams = [torch.cuda.Stream() for _ in range(3)]
    win = native.sf_window_create([[native.make_tensor(*t) for t in s_] for s_ in slots], *streams)
    hl = native.host_layers([[native.make_tensor(*t) for t in L] for L in host])
    steps = (ctypes.c_int64 * n_phys)()
    hp = native.hparams(**HP)
    # warm-up: one visit per physical layer
    native.sf_slide_window_step(win, hl, list(range(n_phys)), hp, steps)
    win.sync()
    # stage times of one visit, each alone (for the overlap efficiency): the
    # fastest of three timings of each, so the efficiency is taken against
    # the best each stage does by itself
    L0, S0 = host[0], slots[0]

    def timed(stream, fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    def h2d():
        for h, d in zip(L0, S0):
            for k in range(4):
                d[k].copy_(h[k], non_blocking=True)

    def upd():
        native.sf_adamw_layer_step([native.make_tensor(*d) for d in S0], hp, 1, streams[1])

    def d2h():
        for h, d in zip(L0, S0):
            for k in (1, 2, 3, 4):
                h[k].copy_(d[k], non_blocking=True)

    t_h2d = min(timed(streams[0], h2d) for _ in range(3))
    t_upd = min(timed(streams[1], upd) for _ in range(3))
    t_d2h = min(timed(streams[2], d2h) for _ in range(3))
    order = [v % n_phys for v in range(n_visits)]
    barrier(world)
    clk = Clocks(bus_id_of_current_device())
    with clk:
        t0 = time.perf_counter()
        native.sf_slide_window_step(win, hl, order, hp, steps)
        win.sync()
        wall = time.perf_counter() - t0
    barrier(world)
    per_layer = synth.layer_numel(layer)
    win.close()
    del host, slots
    release_pinned()
    torch.cuda.empty_cache()
    return dict(wall_s=wall, visits=n_visits, params_per_visit=per_layer, setup_s=setup_s,
                t_h2d_ms=t_h2d, t_update_ms=t_upd, t_d2h_ms=t_d2h, clocks=clk.summary(), steps=list(steps))


def mistral_summary(r, world):
    """The Mistral-Large window's numbers: rate, link GB/s each way, overlap efficiency, update alone."""
    wall = max_over_ranks(r["wall_s"], world)
    params = world * r["params_per_visit"] * r["visits"]
    link_bytes = 14 * r["params_per_visit"] * r["visits"]
    bound = max(r["t_h2d_ms"], r["t_update_ms"], r["t_d2h_ms"])
    peak, kind = measured_peak_hbm()
    upd_gbs = ADAM_BYTES_PER_PARAM * r["params_per_visit"] / (r["t_update_ms"] / 1e3) / 1e9
    return {
        "workload": "Mistral-Large-123B layer (hidden 12288, 96 q / 8 kv heads of 128, SwiGLU FFN 28672; "
                    "1,384,144,896 params); 4 layers in pinned host memory (88.6 GB), 2 device slots, 88 visits "
                    "cycling layers 0..3 (22 updates per layer); 3 streams",
        "value": params / wall, "unit": "params/s", "ms_per_sweep": wall * 1e3, "visits": r["visits"],
        "h2d_bytes_per_sweep": link_bytes, "d2h_bytes_per_sweep": link_bytes,
        "link": {"h2d_GBps": link_bytes / wall / 1e9, "d2h_GBps": link_bytes / wall / 1e9,
                 "one_visit_alone_ms": {"h2d": r["t_h2d_ms"], "update": r["t_update_ms"], "d2h": r["t_d2h_ms"]},
                 "overlap_efficiency": r["visits"] * bound / 1e3 / wall},
        "update_alone": {"kernel": "adamw_bulk_kernel", "GBps": upd_gbs, "frac_of_hbm_peak": upd_gbs / peak,
                         "peak": peak, "peak_kind": kind},
        "clocks": r["clocks"], "setup_s": r["setup_s"], "steps_per_layer": r["steps"],
    }


def main_window(args, rank, world):
    import torch
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    from layer_optimizer_gb300 import native
    native.load()
    m = mistral_summary(run_mistral_window(args, world), world)
    line = {
        "metric": "params updated/s (layer-sliding window, Mistral-Large-123B layer)",
        "value": m["value"], "unit": "params/s", "n_gpus": world, "steps": 1, "warmup": 1,
        "ms_per_step": m["ms_per_sweep"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (bf16 grad in, bf16 weight out)",
        "data": "synthetic (seeded N(0,1e-3) bf16 grads fixed in the host slots, N(0,0.02) fp32 masters)",
        "config": {"workload": m["workload"], "step": "one 88-visit sweep", "warm-up": "one visit per layer",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gpu_launches": m["visits"],
        "e2e": {"value": m["value"], "unit": "params/s", "h2d_bytes_per_step": m["h2d_bytes_per_sweep"],
                "d2h_bytes_per_step": m["d2h_bytes_per_sweep"],
                "path": "sf_slide_window_step (the measured path itself)"},
        "link": m["link"],
        "roofline": {"bound": "host link", "kernel": "adamw_bulk_kernel (in the window)",
                     "update_alone_GBps": m["update_alone"]["GBps"],
                     "update_frac_of_hbm_peak": m["update_alone"]["frac_of_hbm_peak"],
                     "peak": m["update_alone"]["peak"], "peak_kind": m["update_alone"]["peak_kind"]},
        "clocks": m["clocks"], "setup_s": m["setup_s"], "steps_per_layer": m["steps_per_layer"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


LLAMA_CFG = ("LLaMA-2-7B: 32 layers (hidden 4096, 32 heads, SwiGLU FFN 11008) + embedding + LM head (vocab "
             "32000) + final norm = 6,738,415,616 params; bf16 grads, fp32 master/m/v resident in HBM; one fused "
             "AdamW launch per group in sliding order (head, norm, layers 31..0, embedding)")
OPT_CFG = ("OPT-1.3B stack: 24 layers x 50,339,840 params (hidden 2048, FFN 8192, QKV/O/FC1/FC2 + 2 LayerNorms), "
           "one fused AdamW launch per layer")


def opt13_sub(args, world):
    """The OPT-1.3B stack: resident rate and roofline, and its window form with every array on the host."""
    groups = workload_groups("opt-1.3b", args.layers)
    res = run_resident(args, world, groups)
    out = {"workload": OPT_CFG, "params_per_step": res["params_per_step"], "steps": args.steps,
           "clocks": res["clocks"], "l2": "inputs larger than L2 (1.41 GB per launch)"}
    out.update(resident_summary(res, args, world))
    out["unit"] = "params/s"
    if not args.no_e2e and world > 1:
        out["e2e_window"] = {"skipped": "every array of the stack in pinned host memory (19.3 GB per rank): "
                                        "run in the single-GPU line only"}
    elif not args.no_e2e:
        e = run_e2e(args, world)
        wall = max_over_ranks(e["wall_s"], world)
        out["e2e_window"] = {
            "value": world * e["params_per_step"] * args.steps / wall, "unit": "params/s",
            "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
            "path": "sf_slide_window_step: 24 pinned host layers (flat per-array buffers, every array on the host), "
                    "3 device slots, 3 streams",
            "link_GBps_each_way": e["h2d"] * args.steps / wall / 1e9,
            "same_buffers_plain_copies_GBps_each_way": e["raw_copy_GBps_each_way"]}
        try:
            out["e2e_window"]["link_probe"] = link_probe()
        except Exception as ex:
            out["e2e_window"]["link_probe"] = {"error": str(ex)[:200]}
        release_pinned()
    return out


def main_ours(args, rank, world):
    import torch
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    from layer_optimizer_gb300 import native
    native.load()
    llama = args.workload == "llama2-7b"
    groups = workload_groups(args.workload, args.layers)
    # host memory before any rank pins anything: the legs that pin host
    # buffers on every rank must fit all ranks of this node at once
    avail = host_mem_available()
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", world))
    params = sum(n for g in groups for _, n in g)
    e2e_pinned = params * 4 if llama else params * 16          # bf16 grads + weights; or every array
    run_e2e_leg = not args.no_e2e and (world == 1 or pinned_leg_fits(e2e_pinned, local_ranks, avail))
    res = run_resident(args, world, groups, keep=llama and run_e2e_leg)
    summ = resident_summary(res, args, world)
    if llama:
        metric = "params updated/s (fused AdamW, LLaMA-2-7B full step)"
        cfg = {"workload": LLAMA_CFG, "groups": len(groups), "params_per_step": res["params_per_step"],
               "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
               "l2": "inputs larger than L2 (up to 4.1 GB per launch)"}
    else:
        metric = "params updated/s (fused AdamW, OPT-1.3B stack)"
        cfg = {"workload": OPT_CFG, "layers": args.layers, "params_per_step": res["params_per_step"],
               "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
               "l2": "inputs larger than L2 (1.41 GB per launch)"}
    line = {
        "metric": metric,
        "value": summ["value"],
        "unit": "params/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": summ["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 (bf16 grad in, bf16 weight out)",
        "data": "synthetic (seeded N(0,1e-3) bf16 grads, N(0,0.02) fp32 masters)",
        "config": cfg,
        "gpu_launches": res["launches"],
        "kernels_per_step": res["kernels_per_step"],
        "roofline": summ["roofline"],
        "clocks": res["clocks"],
    }
    if not args.no_e2e and not run_e2e_leg:
        line["e2e"] = {"skipped": f"needs {e2e_pinned / 1e9:.1f} GB of pinned host memory on each of "
                                  f"{local_ranks} ranks; {(avail or 0) / 1e9:.1f} GB available on this node"}
    elif not args.no_e2e:
        if llama:
            e = run_e2e_states_resident(args, world, groups, res.pop("layers"), res["steps_done"])
            wall = max_over_ranks(e["wall_s"], world)
            line["e2e"] = {"value": world * e["params_per_step"] * args.steps / wall, "unit": "params/s",
                           "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                           "path": "sf_slide_window_step with master/m/v resident in HBM: each step every "
                                   "group's bf16 gradients come from pinned host memory and its bf16 weights go "
                                   "back (3 device slots, 3 streams)",
                           "link_GBps_each_way": e["h2d"] * args.steps / wall / 1e9}
        else:
            e = run_e2e(args, world)
            wall = max_over_ranks(e["wall_s"], world)
            line["e2e"] = {"value": world * e["params_per_step"] * args.steps / wall, "unit": "params/s",
                           "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                           "path": "sf_slide_window_step: 24 pinned host layers (flat per-array buffers), 3 device "
                                   "slots, 3 streams",
                           "link_GBps_each_way": e["h2d"] * args.steps / wall / 1e9,
                           "same_buffers_plain_copies_GBps_each_way": e["raw_copy_GBps_each_way"]}
            release_pinned()
    res.pop("layers", None)
    torch.cuda.empty_cache()
    if llama:
        try:
            line["opt13"] = opt13_sub(args, world)
        except Exception as ex:
            line["opt13"] = {"error": str(ex)[:300]}
        if not args.no_c5 and world > 1:
            line["mistral_window"] = {"skipped": "the Mistral-Large window pins 88.6 GB of host memory per rank; "
                                                 "it runs in the single-GPU line only"}
        elif not args.no_c5:
            try:
                line["mistral_window"] = mistral_summary(run_mistral_window(args, world), world)
            except Exception as ex:
                line["mistral_window"] = {"error": str(ex)[:300]}
    if not args.no_lsp and rank == 0:
        try:
            line["lsp"] = run_lsp(args)
        except Exception as ex:  # the line still prints; the failure is recorded on it
            line["lsp"] = {"error": str(ex)[:300]}
    if not args.no_lce and rank == 0:
        try:
            line["lce"] = run_lce(args)
        except Exception as ex:
            line["lce"] = {"error": str(ex)[:300]}
    if not args.no_cpu and rank == 0:
        line["host_update"] = host_update_rate()
        # the oracle beside the other two workloads (bounded samples)
        if isinstance(line.get("lsp"), dict) and "error" not in line["lsp"]:
            line["lsp"]["cpu_oracle"] = oracle_lsp_chain_rate()
        if isinstance(line.get("lce"), dict) and "error" not in line["lce"]:
            line["lce"]["cpu_oracle"] = oracle_lce_rate()
    if not args.no_cpu and rank == 0:
        v, done, el = oracle_params_per_s()
        line["cpu_baseline"] = {"value": v, "unit": "params/s", "cores": 1, "kind": "oracle",
                                "sample": f"fp64 numpy AdamW on 2^21-param chunks of a "
                                          f"{'LLaMA-2-7B q' if llama else 'OPT-1.3B'} tensor, {done} params in "
                                          f"{el:.1f} s (elementwise numpy: one thread)"}
        line["cpu_baseline"].update(cpu_context())
    if rank == 0:
        print(json.dumps(line), flush=True)


def main_reference(args, rank, world):
    if rank != 0:
        return
    steps_v = []
    total_done, total_el = 0, 0.0
    for i in range(args.warmup + args.steps):
        v, done, el = oracle_params_per_s(budget_s=1e9, chunk=1 << 21, max_steps=1)
        if i >= args.warmup:
            total_done += done
            total_el += el
    value = total_done / total_el
    line = {
        "impl": "reference",
        "metric": ("params updated/s (fused AdamW, LLaMA-2-7B full step)" if args.workload == "llama2-7b"
                   else "params updated/s (fused AdamW, OPT-1.3B stack)"),
        "value": value, "unit": "params/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": (LLAMA_CFG if args.workload == "llama2-7b" else OPT_CFG) +
                   " (bounded sample: one 2^21-param chunk per step)"},
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle",
                         "sample": "one 2^21-param chunk of a weight tensor per step"},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.profile_small:
        args.workload = "opt-1.3b"
        args.layers, args.steps, args.warmup = 1, 1, 1
        args.no_e2e = args.no_lsp = args.no_cpu = args.no_lce = True
    if args.profile_lce:
        import torch
        from layer_optimizer_gb300 import native
        native.load()
        print(json.dumps({"profile_lce": run_lce(args, N=2048, V=32000)}))
        return
    if args.profile_lsp:
        import torch
        from layer_optimizer_gb300 import native
        native.load()
        args.warmup = 1
        print(json.dumps({"profile_lsp": run_lsp(args, matrices=[("q", 4096, 4096)])}))
        return
    rank, world = dist_init(args)
    if args.impl == "reference":
        main_reference(args, rank, world)
    elif args.workload == "mistral-window":
        main_window(args, rank, world)
    else:
        main_ours(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

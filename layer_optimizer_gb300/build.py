"""Builds the C-ABI shared library ``libsfopt.so`` for sm_103a with nvcc.

Every translation unit under ``csrc/`` is compiled in parallel into
``_build/`` at the repository root, then linked into
``layer_optimizer_gb300/libsfopt.so`` (in-tree, git-ignored).  A unit is
recompiled when its source, any header, or the flags changed.  No CMake.

Usage: ``python -m layer_optimizer_gb300.build [--force] [-v]``
"""

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libsfopt.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O3,-Wall",
          "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin on PATH)")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sorted(hs)


def _stamp(src, flags):
    h = hashlib.sha256()
    for p in [src] + _headers():
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(flags).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


# Per-file extra flags: the host AdamW must not contract a*b+c into an FMA
# where the device kernel does not, so both give the same bits.
FILE_FLAGS = {"host_adamw.cpp": ["-Xcompiler", "-ffp-contract=off"]}


def _compile(nvcc, src, flags, verbose):
    flags = list(flags) + FILE_FLAGS.get(os.path.basename(src), [])
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    stamp_file = obj + ".stamp"
    stamp = _stamp(src, flags)
    if os.path.exists(obj) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read() == stamp:
                return obj, False
    cmd = [nvcc] + ARCH + flags + ["-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout.strip() or r.stderr.strip()):
        print(r.stdout + r.stderr, flush=True)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return obj, True


def build(force=False, verbose=False, extra_flags=()):
    """Compile and link libsfopt.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    flags = CFLAGS + list(extra_flags)
    if force:
        for f in os.listdir(BUILD):
            if f.endswith(".stamp"):
                os.remove(os.path.join(BUILD, f))
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s, flags, verbose), srcs))
    objs = [o for o, _ in results]
    changed = any(c for _, c in results)
    if changed or not os.path.exists(LIB) or force:
        tmp = LIB + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

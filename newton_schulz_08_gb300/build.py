"""Builds libmuon.so in-tree with nvcc for sm_103a (no CMake).

Each .cu translation unit is compiled in parallel to an object file, then the
objects are linked into ``newton_schulz_08_gb300/lib/libmuon.so`` with the
CUDA runtime linked statically.  Run ``python -m newton_schulz_08_gb300.build``.
"""

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libmuon.so")
DEBUG_LIB = os.path.join(LIBDIR, "libmuon_debug.so")  # device-side checks (MUON_DEBUG)
SOURCES = ["muon_capi.cu", "elementwise.cu", "ns_gemm.cu", "fp8.cu", "noalloc.cu", "partition.cu", "adam.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand) and not shutil.which(cand):
        raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")
    return cand


def flags():
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _compile(src, extra, obj_dir):
    out = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", out] + flags() + extra
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return out, r.stderr


def _link(objs, lib):
    tmp = lib + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-lcudart_static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(verbose=False, extra=(), debug=True):
    """Builds libmuon.so and, with debug=True, libmuon_debug.so (the same
    sources with -DMUON_DEBUG), every translation unit in parallel."""
    os.makedirs(LIBDIR, exist_ok=True)
    extra = list(extra)
    variants = [(OBJ, extra, LIB)]
    if debug:
        variants.append((OBJ + "_debug", extra + ["-DMUON_DEBUG"], DEBUG_LIB))
    jobs = []
    for obj_dir, ex, _ in variants:
        os.makedirs(obj_dir, exist_ok=True)
        jobs += [(src, ex, obj_dir) for src in SOURCES]
    with concurrent.futures.ThreadPoolExecutor(len(jobs)) as pool:
        results = list(pool.map(lambda j: _compile(*j), jobs))
    if verbose:
        for _, err in results:
            if err.strip():
                print(err, file=sys.stderr)
    for k, (_, _, lib) in enumerate(variants):
        _link([o for o, _ in results[k * len(SOURCES):(k + 1) * len(SOURCES)]], lib)
    return LIB


if __name__ == "__main__":
    verbose = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(verbose=verbose or bool(extra), extra=extra))

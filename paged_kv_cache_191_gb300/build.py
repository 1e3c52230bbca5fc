"""Build libpagedkv.so in-tree with nvcc (sm_103a only).

Usage: ``python -m paged_kv_cache_191_gb300.build [--force]``.  Translation
units compile in parallel; the shared library links the CUDA runtime
statically so it loads without a GPU (host-only calls such as the block
manager work anywhere).
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedkv.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
          "--expt-relaxed-constexpr"]
SOURCES = ["decode.cu", "decode_static.cu", "prefill.cu", "cache_ops.cu", "api.cpp", "allocator.cpp", "scheduler.cpp",
           "serve.cpp", "segments.cpp"]
HEADERS = ["device_common.cuh", "pa_internal.h", "kv_map.h"]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv.so")
    return exe


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "pagedkv.h"), __file__]
    return any(os.path.getmtime(p) > t for p in deps)


def _compile(src, extra):
    obj = os.path.join(BUILD, src + ".o")
    cmd = [nvcc(), *ARCH, *COMMON, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force=False, verbose=False, extra=()):
    """Compile and link libpagedkv.so; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, list(extra)), SOURCES))
    if verbose:
        for (_, err), src in zip(results, SOURCES):
            if err.strip():
                print(f"--- {src}\n{err}", file=sys.stderr)
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static",
           *[o for o, _ in results], "-o", tmp, "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    args = sys.argv[1:]
    extra = [a for a in args if a.startswith("-D")]  # tuning macros, e.g. -DPA_RING_KB=32
    if "--ptxas-v" in args:
        extra += ["-Xptxas", "-v"]
    print(build(force="--force" in args or bool(extra), verbose="--ptxas-v" in args, extra=extra))

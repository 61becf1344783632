"""Builds libw4g128.so in-tree for sm_103a with nvcc (no cmake, no torch
extension machinery): each translation unit is compiled in parallel, then
linked into one shared library with the CUDA runtime linked statically."""
import concurrent.futures
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libw4g128.so")
# The same sources with -DW4G128_DEBUG: every global access the kernels derive
# from the schedule is range-checked, a failed check is recorded in the status
# word and the access skipped (for tests; slower, never used by the product).
DEBUG_BUILD = os.path.join(BUILD, "debug")
LIB_DEBUG = os.path.join(BUILD, "libw4g128_debug.so")

SOURCES = ["w4g128_api.cu", "w4g128_pack.cu", "w4g128_stream.cu", "w4g128_probe.cu", "w4g128_noalloc.cu",
           "w4g128_quant.cu", "w4g128_selftest.cu", "w4g128_hostio.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC]


def _headers():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, extra, outdir=BUILD):
    obj = os.path.join(outdir, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src)] + _headers()
    if _stale(obj, deps) or extra:
        cmd = ["nvcc", "-c", os.path.join(CSRC, src), "-o", obj] + ARCH + FLAGS + list(extra)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(extra_flags=(), force=False, verbose=False, debug=False):
    """Compile (if stale) and return the path of libw4g128.so (debug: of
    libw4g128_debug.so, the range-checked build)."""
    outdir, lib = (DEBUG_BUILD, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(outdir, exist_ok=True)
    extra = list(extra_flags)
    flags = extra + (["-DW4G128_DEBUG"] if debug else [])
    if force and os.path.exists(lib):
        os.remove(lib)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, flags, outdir) if not debug else _compile_debug(s, flags, outdir),
                           SOURCES))
    if _stale(lib, objs) or extra:
        # -fvisibility=hidden keeps internal symbols out; the extern "C" API is
        # exported by the W4G128_API attribute on its declarations.
        cmd = ["nvcc", "-shared", "-o", lib] + objs + ARCH + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(lib, file=sys.stderr)
    return lib


def _compile_debug(src, flags, outdir):
    """Like _compile, but the define alone does not make a stale object."""
    obj = os.path.join(outdir, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src)] + _headers()
    if _stale(obj, deps) or len(flags) > 1:
        cmd = ["nvcc", "-c", os.path.join(CSRC, src), "-o", obj] + ARCH + FLAGS + list(flags)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


if __name__ == "__main__":
    build(verbose=True)
    build(verbose=True, debug=True)

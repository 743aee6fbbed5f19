"""Build the CUDA library in-tree for sm_103a.

Each ``csrc/*.cu`` is compiled in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo`` and linked into
``_build/libnvfp4draft.so`` (CUDA runtime linked statically, so the library
is self-contained; it shares the process's primary CUDA context).
"""
import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libnvfp4draft.so")
# Variant with device-side bounds checks on every access (see common.cuh).
DEBUG_LIB = os.path.join(OUT, "libnvfp4draft_debug.so")
# Test variant whose kernels withhold one copy, so a bounded wait runs out (the
# timeout tests load it; see NVFP4_TEST_WITHHOLD in common.cuh).  Built with
# the library.
WITHHOLD_LIB = os.path.join(OUT, "libnvfp4draft_withhold.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
         "--expt-relaxed-constexpr"]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def _stale(srcs, target):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    deps = srcs + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "nvfp4draft.h"),
                                                              __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False, extra=(), debug=False, withhold=False):
    if not debug and not withhold:
        # the library and its timeout-test variant, side by side
        with cf.ThreadPoolExecutor(2) as ex:
            fw = ex.submit(build, force, verbose, extra, False, True)
            lib = _build_one(force, verbose, extra, False, False)
            fw.result()
        return lib
    return _build_one(force, verbose, extra, debug, withhold)


def _build_one(force, verbose, extra, debug, withhold):
    os.makedirs(OUT, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    lib = DEBUG_LIB if debug else (WITHHOLD_LIB if withhold else LIB)
    tag = "_debug" if debug else ("_withhold" if withhold else "")
    if debug:
        extra = tuple(extra) + ("-DNVFP4_DEBUG_BOUNDS",)
    if withhold:
        extra = tuple(extra) + ("-DNVFP4_TEST_WITHHOLD",)
    if not force and not _stale(srcs, lib):
        return lib
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(OUT, os.path.basename(src)[:-3] + tag + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))

"""Build libpw.so in-tree for sm_103a (nvcc, one object per .cu, compiled in parallel)."""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpw.so")
# the traced variant (GEMM pipeline stamps, -DPW_TRACE): its own objects and library
OBJ_TRACE = os.path.join(PKG, "_build_trace")
LIB_TRACE = os.path.join(PKG, "libpw_trace.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src, extra, objdir=OBJ):
    obj = os.path.join(objdir, os.path.basename(src).replace(".cu", ".o"))
    if os.path.exists(obj) and os.path.getmtime(obj) >= _newest_input(src):
        return obj, ""
    cmd = [nvcc()] + ARCH + FLAGS + extra + ["-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), res.stderr))
    return obj, res.stderr


def _newest_input(src):
    deps = [src, os.path.join(ROOT, "include", "pw.h")] + glob.glob(os.path.join(CSRC, "*.cuh"))
    return max(os.path.getmtime(d) for d in deps)


def build(verbose=False, extra=(), trace=False):
    """Build libpw.so, or with `trace` libpw_trace.so (the same sources with
    -DPW_TRACE, for pw_debug_gemm_trace); returns the library's path."""
    objdir, lib = (OBJ_TRACE, LIB_TRACE) if trace else (OBJ, LIB)
    extra = list(extra) + (["-DPW_TRACE"] if trace else [])
    os.makedirs(objdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, objdir), srcs))
    if verbose:
        for obj, err in results:
            if err:
                print(err, file=sys.stderr)
    objs = [o for o, _ in results]
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", lib] + objs
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), res.stderr))
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, trace="--trace" in sys.argv))

"""Build the in-tree CUDA library ``liblamb_gb300.so`` for sm_103a.

Three translation units are compiled in parallel with nvcc and linked into one
shared object with the CUDA runtime linked statically, so the library loads
(and its symbols can be inspected) on a machine without a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblamb_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["lamb_kernels.cu", "lamb_api.cpp", "lamb_plan.cpp", "lamb_noalloc.cu",
           "lamb_ptrs.cu"]
HEADERS = [os.path.join(INCLUDE, "lamb.h"), os.path.join(CSRC, "lamb_internal.h")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the LAMB library needs the CUDA toolkit to build")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, defines=(), lib: str = LIB) -> str:
    """Compile the library if any source is newer than it; return its path.

    ``defines`` (e.g. ``["LAMB_TEST_APPLY_REPORTS_WAIT_ERROR=1"]``) and ``lib``
    build a variant elsewhere, for tests that need a build-time hook; the
    default builds the library itself."""
    if not force and lib == LIB and not defines and not _stale():
        return LIB
    nvcc = _nvcc()
    build_dir = BUILD if lib == LIB else lib + ".build"
    os.makedirs(build_dir, exist_ok=True)
    common = ["-std=c++17", "-O3", "-I", INCLUDE, "-I", CSRC, "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-Xcompiler", "-Wall"]
    common += ["-D" + d for d in defines]

    def compile_one(src):
        obj = os.path.join(build_dir, src + ".o")
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + common
        if src.endswith(".cu"):
            cmd += ARCH + ["-lineinfo", "-Xptxas", "-v" if verbose else "-O3"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stderr

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", "-o", tmp] + [o for o, _ in results] + ARCH + ["-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

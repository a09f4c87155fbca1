"""Build the C-ABI library `libkvc.so` in-tree with nvcc for sm_103a.

Each translation unit under `csrc/` compiles in parallel to `_build/`, then links into
`_lib/libkvc.so`. A rebuild happens only when a source or header is newer than the library.

The same sources built with KVC_DEBUG_BOUNDS give `_lib/libkvc_debug.so` (objects in
`_build_debug/`): guard bands around every buffer the library allocates and an index check on every
global store of every kernel, the stand-in for a memory checker in tests (the binding loads it when
the environment sets KVC_DEBUG_BOUNDS=1).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libkvc.so")
LIB_DEBUG = os.path.join(LIBDIR, "libkvc_debug.so")
DEBUG_FLAGS = ["-DKVC_DEBUG_BOUNDS"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps() + [os.path.abspath(__file__)])


def _compile(nvcc, src, outdir, extra):
    obj = os.path.join(outdir, os.path.basename(src) + ".o")
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _link(nvcc, objs, lib):
    tmp = lib + ".tmp"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = True) -> str:
    """Compile every CUDA/C++ source for sm_103a and link `_lib/libkvc.so` (and, with `debug`,
    `_lib/libkvc_debug.so`, in the same parallel pass); returns the release library's path."""
    targets = [(LIB, BUILD, list(extra_flags))]
    if debug:
        targets.append((LIB_DEBUG, BUILD_DEBUG, list(extra_flags) + DEBUG_FLAGS))
    targets = [t for t in targets if force or not up_to_date(t[0])]
    if not targets:
        return LIB
    nvcc = _nvcc()
    os.makedirs(LIBDIR, exist_ok=True)
    for _, outdir, _ in targets:
        os.makedirs(outdir, exist_ok=True)
    srcs = _sources()
    jobs = [(src, outdir, flags) for _, outdir, flags in targets for src in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda j: _compile(nvcc, *j), jobs))
    if verbose:
        for _, err in results:
            if err.strip():
                print(err, file=sys.stderr)
    for k, (lib, _, _) in enumerate(targets):
        _link(nvcc, [o for o, _ in results[k * len(srcs):(k + 1) * len(srcs)]], lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else []))

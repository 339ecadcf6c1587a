"""Builds libtq.so (the C-ABI library) in-tree with nvcc for sm_103a.

Every translation unit is compiled in parallel; objects live in ``_build/``
next to this file and ``libtq.so`` lands in the package directory.  ptxas
resource usage (registers, spills, shared memory) of each kernel is kept in
``_build/ptxas.log``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INC = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build", platform.machine())   # objects per host architecture
LIB = os.path.join(PKG, "libtq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

# Build variants: the library (default) and the profiling build that records the decode
# and combine kernels' phase timeline (-DTQ_TIMELINE, libtq_timeline.so).
VARIANTS = {None: ([], "", "libtq.so"), "timeline": (["-DTQ_TIMELINE"], "-timeline", "libtq_timeline.so")}


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or "/usr/local/cuda"
    if not os.path.exists(os.path.join(home, "bin", "nvcc")):
        nv = shutil.which("nvcc")
        if nv:
            home = os.path.dirname(os.path.dirname(os.path.realpath(nv)))
    return home


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(INC, "tq.h")]


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(f) > t for f in [src] + _headers())


def _compile(src: str, cuda: str, build_dir: str, defs: list) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    if not _stale(obj, src):
        return obj, ""
    nvcc = os.path.join(cuda, "bin", "nvcc")
    common = ["-O3", "-std=c++17", "-I", INC, "-I", CSRC, "-Xcompiler", "-fPIC", *defs]
    if src.endswith(".cu"):
        cmd = [nvcc, *ARCH, "-lineinfo", "--expt-relaxed-constexpr", "-Xptxas", "-v", *common,
               "-c", src, "-o", obj]
    else:
        cmd = [nvcc, *common, "-x", "c++", "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, variant: str | None = None) -> str:
    """Compile every csrc/*.cu and *.cpp and link the library of `variant` (None: libtq.so);
    returns its path."""
    cuda = _cuda_home()
    defs, suffix, libname = VARIANTS[variant]
    build_dir = BUILD + suffix
    lib_path = os.path.join(PKG, libname)
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, cuda, build_dir, defs), srcs))
    objs = [o for o, _ in results]
    logs = [log for _, log in results if log]
    if logs:
        with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
            f.write("\n".join(logs))
    stamp = os.path.join(build_dir, "libtq.stamp")     # the library was linked from this architecture's objects
    fresh = os.path.exists(lib_path) and os.path.exists(stamp) and \
        all(os.path.getmtime(o) <= os.path.getmtime(lib_path) for o in objs)
    if not fresh:
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [os.path.join(cuda, "bin", "nvcc"), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath," + os.path.join(cuda, "lib64")]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
        with open(stamp, "w") as f:
            f.write(lib_path + "\n")
    if verbose:
        print(lib_path)
    return lib_path


E2E_SRC = os.path.join(CSRC, "e2e", "tq_e2e_loop.cpp")
E2E_LIB = os.path.join(PKG, "libtq_e2e.so")


def build_e2e(verbose: bool = False) -> str:
    """The benchmark's end-to-end driver (libtq_e2e.so): a C loop over the public C ABI,
    linked against libtq.so; returns its path."""
    lib = build(verbose=verbose)
    cuda = _cuda_home()
    stamp = os.path.join(BUILD, "libtq_e2e.stamp")
    if os.path.exists(E2E_LIB) and os.path.exists(stamp) and \
            os.path.getmtime(E2E_LIB) >= max(os.path.getmtime(E2E_SRC), os.path.getmtime(lib)):
        return E2E_LIB
    tmp = E2E_LIB + f".tmp{os.getpid()}"
    cmd = [os.path.join(cuda, "bin", "nvcc"), "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-I", INC,
           "-x", "c++", E2E_SRC, "-o", tmp, "-L", PKG, "-ltq", "-cudart", "shared",
           "-Xlinker", "-rpath,$ORIGIN", "-Xlinker", "-rpath," + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, E2E_LIB)
    with open(stamp, "w") as f:
        f.write(E2E_LIB + "\n")
    return E2E_LIB


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, variant="timeline" if "--timeline" in sys.argv else None)

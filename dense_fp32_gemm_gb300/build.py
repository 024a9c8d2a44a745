"""Build the CUDA library libsgemm_gb300.so in-tree for sm_103a.

Each .cu file under csrc/ is compiled on its own (in parallel) and the objects
are linked into ``_lib/libsgemm_gb300.so`` with the CUDA runtime linked
statically, so the library loads on any machine with the driver installed.
Only the functions declared in include/sgemm_gb300.h are exported.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB_NAME = "libsgemm_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "--expt-relaxed-constexpr", "-O3", "-lineinfo",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-Xptxas", "-v"] + ARCH


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h*")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.inc")) + glob.glob(os.path.join(HERE, "..", "include", "*.h"))


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(f) > t for f in [src] + _headers())


def build(verbose: bool = False, jobs: int | None = None) -> str:
    """Compile (what changed) and link; returns the library path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    tool = nvcc()
    srcs = sources()
    objs = [os.path.join(OUT_DIR, os.path.basename(s)[:-3] + ".o") for s in srcs]
    logs = {}

    def compile_one(pair):
        src, obj = pair
        if not _stale(obj, src):
            return
        cmd = [tool] + NVCC_FLAGS + ["-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        logs[src] = r.stdout + r.stderr
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr[-4000:]}")
        os.replace(obj + ".tmp", obj)

    n = jobs or min(len(srcs), os.cpu_count() or 1)
    with ThreadPoolExecutor(max(1, n)) as ex:
        list(ex.map(compile_one, zip(srcs, objs)))
    if verbose:
        for src, log in sorted(logs.items()):
            print(f"== {os.path.basename(src)}\n{log}", file=sys.stderr)
    lib_stale = not os.path.exists(LIB_PATH) or any(
        os.path.getmtime(o) > os.path.getmtime(LIB_PATH) for o in objs)
    if lib_stale:
        tmp = LIB_PATH + ".tmp"
        subprocess.check_call([tool, "-shared", "-cudart", "static"] + ARCH + objs + ["-o", tmp])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))

"""Build libkvq.so in-tree with nvcc for sm_103a (GB300).

Compiles every ``csrc/*.cu`` translation unit in parallel, then links one
shared library next to this file: ``libkvq.so``, or with ``debug=True``
``libkvq_debug.so``, the same kernels compiled with ``KVQ_DEBUG=1`` so that
their global-memory indices are checked (a failed check reports
KVQ_ERR_BOUNDS and skips the access; the tests run parity cases on it).  The CUDA runtime is linked statically and
the driver is reached through ``cudaGetDriverEntryPointByVersion``, so the
library loads on machines without a GPU driver (its symbols can be checked
there; compute calls need a GB300).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libkvq.so")
OUT_DEBUG = os.path.join(HERE, "libkvq_debug.so")
BUILD = os.path.join(HERE, "_build")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, extra, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(verbose_ptxas: bool = False, debug: bool = False) -> str:
    build_dir, out = (BUILD_DEBUG, OUT_DEBUG) if debug else (BUILD, OUT)
    os.makedirs(build_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if debug:
        extra += ["-DKVQ_DEBUG=1"]
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), srcs))
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))

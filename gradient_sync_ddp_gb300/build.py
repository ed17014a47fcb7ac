"""Build libddp_sync.so in-tree for sm_103a.

Each translation unit compiles in parallel (nvcc for .cu, g++ for .cpp) into
``_build/``; the objects link into ``libddp_sync.so`` next to this file.  The
device code is compiled for exactly one target, ``sm_103a``, without fast-math
(subnormals kept, IEEE division and square root, no flush-to-zero); the host
code with ``-ffp-contract=off``.

Usage: ``python gradient_sync_ddp_gb300/build.py [--force] [--verbose] [--ptxas]``
(run it by path: importing the package needs the library this builds).
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
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libddp_sync.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
# per-file extra flags: the bit-exact averaging kernels also forbid contraction globally
EXTRA = {"allreduce.cu": ["-fmad=false"]}
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-Wall", "-I", INCLUDE, "-I", CSRC]


def _cuda_home():
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps() + [__file__])


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every translation unit and link the shared library; returns its path."""
    if not force and up_to_date():
        return LIB
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(BUILD, exist_ok=True)
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD, src + ".o")
        path = os.path.join(CSRC, src)
        if src.endswith(".cu"):
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *EXTRA.get(src, [])]
            if ptxas_verbose:
                cmd += ["-Xptxas", "-v"]
            cmd += ["-c", path, "-o", obj]
        else:
            cmd = ["g++", *CXX_FLAGS, "-I", os.path.join(cuda, "include"), "-c", path, "-o", obj]
        jobs.append((cmd, obj))
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        for f in [ex.submit(_run, cmd, verbose or ptxas_verbose) for cmd, _ in jobs]:
            f.result()
    tmp = LIB + ".tmp"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs], "-cudart", "shared",
            "-Xlinker", "-rpath," + os.path.join(cuda, "lib64")]
    _run(link, verbose)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    path = build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
                 ptxas_verbose="--ptxas" in sys.argv)
    print(path)

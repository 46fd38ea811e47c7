"""Build ``libmoe.so`` (the CUDA library behind include/moe.h) in-tree for sm_103a.

    python -m sparse_mixture_experts_61_b300.build [--force] [--ptxas-log]

Each ``csrc/*.cu`` file is compiled by nvcc in parallel into ``_build/`` and the
objects are linked (with the static CUDA runtime) into
``sparse_mixture_experts_61_b300/libmoe.so``.  Only the ``moe_*`` C symbols are
exported.  ``--ptxas-log`` keeps ptxas's register / spill / shared-memory report
in ``_build/ptxas.log``.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmoe.so")
HEADER = os.path.join(ROOT, "include", "moe.h")

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]
# MOE_NVTX=1: compile in NVTX ranges around moe_forward's stages (rebuild with --force).
if os.environ.get("MOE_NVTX") == "1":
    FLAGS += ["-DMOE_NVTX=1"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + [HEADER]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


def _compile(src: str, ptxas_log: bool):
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj]
    if ptxas_log:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, ptxas_log: bool = False) -> str:
    if not (force or ptxas_log or needs_build()):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_log), sources()))
    objs = [o for o, _ in results]
    if ptxas_log:
        with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
            for _, log in results:
                f.write(log)
    tmp = LIB + ".tmp"
    r = subprocess.run([NVCC, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, ptxas_log="--ptxas-log" in sys.argv))

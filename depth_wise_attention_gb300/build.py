"""Build libattnres.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel into _build/, then
linked into depth_wise_attention_gb300/libattnres.so.  A unit is recompiled
when it, any header it can include, or this script is newer than its object.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libattnres.so")

SOURCES = [
    "attnres_api.cu",
    "kernels_bf16.cu",
    "kernels_bf16_multi.cu",
    "kernels_f32.cu",
    "kernels_f32_multi.cu",
    "kernels_phase2.cu",
    "kernels_phase2_mh.cu",
    "kernels_mma.cu",
    "kernels_bwd_split.cu",
    "kernels_bwd_one.cu",
    "kernels_mma_multi.cu",
    "kernels_bwd.cu",
    "kernels_bwd_mh.cu",
    "kernels_bwd_qg.cu",
    "kernels_merge_bwd.cu",
    "kernels_decode.cu",
    "msar.cu",
    "msar_tile.cu",
    "msar_phase1.cu",
    "msar_phase2.cu",
    "msar_bwd.cu",
    "state_merge_bwd.cu",
]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattnres.so")


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(ROOT, "include", "attnres.h"))
    hs.append(os.path.abspath(__file__))
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if needed) and return the path of libattnres.so."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    headers = _headers()
    jobs = []
    objs = []
    for src in SOURCES:
        cu = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [cu] + headers):
            jobs.append((cu, obj))

    def compile_one(job):
        cu, obj = job
        tmp = obj + f".tmp{os.getpid()}"
        cmd = [nvcc] + FLAGS + ["-c", cu, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(cu)}:\n{r.stderr}")
        os.replace(tmp, obj)
        return os.path.basename(cu)

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for name in ex.map(compile_one, jobs):
                if verbose:
                    print(f"compiled {name}", file=sys.stderr)
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static", "-lrt", "-ldl",
                                                               "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libattnres.so failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

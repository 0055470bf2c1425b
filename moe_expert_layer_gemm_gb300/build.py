"""Builds libmoe_gb300.so from csrc/*.cu for sm_103a with nvcc (translation units compiled in
parallel, then linked).  The library links the CUDA runtime statically and reaches the driver's
tensor-map encoder through the runtime's entry-point query, so it needs no libcuda at link time.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmoe_gb300.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + INCLUDE, "-I" + CSRC]
# Extra nvcc flags (e.g. -D tuning switches); a non-empty value forces a full rebuild.
EXTRA = os.environ.get("MOE_NVCC_EXTRA", "").split()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build the MoE library")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


FLAGS_STAMP = os.path.join(BUILD, "extra_flags.txt")


def build(verbose: bool = False, force: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    # objects built with other extra flags than now are stale too
    prev = open(FLAGS_STAMP).read() if os.path.exists(FLAGS_STAMP) else None
    if prev != " ".join(EXTRA):
        force = True
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "moe_gb300.h"))
    cc = nvcc()
    jobs = []
    objs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or EXTRA or _stale(obj, [src] + headers):
            cmd = [cc, *ARCH, *FLAGS, *EXTRA, "-c", src, "-o", obj]
            if ptxas_info:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            for cmd, p in ex.map(run, jobs):
                if verbose or ptxas_info or p.returncode != 0:
                    sys.stderr.write(" ".join(cmd) + "\n" + p.stdout + p.stderr)
                if p.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {cmd[-3]}")
    if force or EXTRA or jobs or _stale(LIB, objs):
        cmd = [cc, *ARCH, "-shared", "-o", LIB, *objs]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + p.stdout + p.stderr)
            raise RuntimeError("linking libmoe_gb300.so failed")
    with open(FLAGS_STAMP, "w") as f:
        f.write(" ".join(EXTRA))
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, ptxas_info="--ptxas" in sys.argv))

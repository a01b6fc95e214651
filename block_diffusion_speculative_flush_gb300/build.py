"""Builds libdflash.so in-tree from csrc/ with nvcc for sm_103a.

    python -m block_diffusion_speculative_flush_gb300.build [--force]

Translation units compile in parallel; the shared library links the CUDA
runtime statically, so it needs neither torch nor a CUDA runtime on the
library path to load.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
MACHINE = os.uname().machine
BUILD = os.path.join(ROOT, "_build", MACHINE)
LIB = os.path.join(PKG, "libdflash.so")
STAMP = LIB + ".machine"   # which architecture the library was linked for

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    jobs = [(s, o) for s, o in zip(srcs, objs) if force or _stale(o, [s] + hdrs)]

    def compile_one(job):
        s, o = job
        cmd = [NVCC, *ARCH, *FLAGS, "-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return s, r.returncode, r.stdout + r.stderr

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for s, rc, out in ex.map(compile_one, jobs):
                if verbose or rc:
                    sys.stderr.write(out)
                if rc:
                    raise RuntimeError(f"nvcc failed on {os.path.basename(s)}")
    linked_for = open(STAMP).read().strip() if os.path.exists(STAMP) else ""
    if force or jobs or _stale(LIB, objs) or linked_for != MACHINE:
        cmd = [NVCC, *ARCH, "-shared", "-o", LIB, *objs, "-Xlinker", "--no-undefined"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link of libdflash.so failed")
        with open(STAMP, "w") as f:
            f.write(MACHINE + "\n")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

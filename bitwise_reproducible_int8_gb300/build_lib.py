"""Builds librepro.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each .cu translation unit is compiled in parallel into ``_build/`` and linked
into ``librepro.so`` next to this file (CUDA runtime linked statically).
Rebuilds only what changed.  Arithmetic-relevant flags: no FMA contraction,
IEEE division and square root, no global flush-to-zero (the kernels choose
their flushing instruction by instruction).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librepro.so")

SOURCES = ["api.cu", "k_scale.cu", "k_quant.cu", "k_fwd.cu", "k_fwd_tc.cu", "k_bwd.cu", "k_bwd_prefetch.cu", "k_bwd_tma.cu",
           "k_reduce.cu", "k_scale_noalloc.cu", "k_optim.cu", "k_hash.cu", "k_attn_fwd.cu", "k_attn_bwd.cu", "k_selftest.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
    "-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-I" + INCLUDE, "-I" + CSRC,
]


def nvcc() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librepro.so")


def _headers():
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    hdrs = _headers()
    cc = nvcc()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, *hdrs, __file__]):
            cmd = [cc, *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append((src, cmd))

    def run(job):
        name, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return name, cmd, r

    failures = []
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for name, cmd, r in ex.map(run, jobs):
                if verbose and (r.stdout or r.stderr):
                    sys.stderr.write(f"--- {name}\n{r.stdout}{r.stderr}")
                if r.returncode != 0:
                    failures.append(f"{' '.join(cmd)}\n{r.stdout}{r.stderr}")
    if failures:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failures))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

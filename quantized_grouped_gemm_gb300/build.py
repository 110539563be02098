"""Build the sm_103a shared library ``libmoe_gb300.so`` in-tree with nvcc.

Each ``csrc/*.cu`` file is compiled in parallel (``-gencode arch=compute_103a,code=sm_103a``)
and the objects are linked into one shared library exporting the C ABI of ``include/moe.h``.
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
LIB = os.path.join(HERE, "libmoe_gb300.so")
SOURCES = ["api.cu", "route.cu", "ffn.cu", "decode.cu", "decode_fused.cu", "pack.cu", "static_scratch.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
                   *extra]


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src, os.path.join(CSRC, "moe_internal.cuh"), os.path.join(ROOT, "include", "moe.h")]
    return any(os.path.getmtime(d) > os.path.getmtime(obj) for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, defines=(), out: str = None,
          build_dir: str = None) -> str:
    """Compile and link; `defines` (e.g. ["MOE_PF_RAW=8"]) override tuning constants, `out` and
    `build_dir` place a variant library elsewhere."""
    global BUILD, LIB
    saved = (BUILD, LIB)
    if out is not None:
        LIB, BUILD = out, build_dir or (out + ".objs")
        force = True
    try:
        return _build(force, verbose, ptxas_info, [f"-D{d}" for d in defines])
    finally:
        BUILD, LIB = saved


def _build(force, verbose, ptxas_info, dflags):
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        if force or _stale(o, s) or ptxas_info:
            extra = (["-Xptxas", "-v"] if ptxas_info else []) + dflags
            jobs.append((src, [cc, *_flags(extra), "-c", s, "-o", o]))

    def run(job):
        name, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return name, cmd, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for name, cmd, r in ex.map(run, jobs):
                if verbose or ptxas_info or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {name}: {' '.join(cmd)}")
    objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)

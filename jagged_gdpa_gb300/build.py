"""Builds libjgdpa.so in-tree (jagged_gdpa_gb300/_build/) with nvcc for sm_103a.

The forward and backward sources are compiled once per head dimension
(-DJGDPA_HEAD_DIM=32/64/128), and every object is compiled in parallel, then
linked into one shared library with the CUDA runtime linked statically, so
the library loads on a machine without a GPU driver (the CUDA calls fail
there, the symbols are still present).

Two libraries are built:
  _build/libjgdpa.so        the product: GELU/SiLU through the hardware tanh
  _build/alu/libjgdpa.so    the same library with every GELU/SiLU element of
                            the forward and backward kernels on the ALU-only
                            polynomial route (JGDPA_FWD_ALU_CHUNKS=4,
                            JGDPA_BWD_ALU_GROUPS=4), so that route's kernel
                            instantiations are compiled and parity-tested
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libjgdpa.so")
HEAD_DIMS = (32, 64, 128)
SOURCES = ["api.cu", "sched.cu"]                 # compiled once
PER_DIM_SOURCES = ["fwd.cu", "fwd_shortq.cu", "bwd.cu", "bwd_shortq.cu"]  # compiled once per head dimension
HEADERS = ["act.cuh", "common.cuh", "ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]
VARIANTS = {
    None: [],
    "alu": ["-DJGDPA_FWD_ALU_CHUNKS=4", "-DJGDPA_BWD_ALU_GROUPS=4"],
}


def lib_path(variant: str | None = None) -> str:
    return LIB if variant is None else os.path.join(BUILD, variant, "libjgdpa.so")


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libjgdpa.so")
    return cand


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src, __file__] + [os.path.join(CSRC, h) for h in HEADERS] + \
        [os.path.join(HERE, "..", "include", "jgdpa.h")]
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def _compile_jobs(cc: str, force: bool):
    """(command, object) per object file of every variant; shared objects once."""
    jobs, objs = [], {v: [] for v in VARIANTS}
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, s.replace(".cu", ".o"))
        for v in VARIANTS:
            objs[v].append(obj)
        if force or _stale(obj, src):
            jobs.append([cc, *ARCH, *FLAGS, "-c", src, "-o", obj])
    for v, vflags in VARIANTS.items():
        out_dir = BUILD if v is None else os.path.join(BUILD, v)
        os.makedirs(out_dir, exist_ok=True)
        for s in PER_DIM_SOURCES:
            src = os.path.join(CSRC, s)
            for d in HEAD_DIMS:
                obj = os.path.join(out_dir, s.replace(".cu", f"_d{d}.o"))
                objs[v].append(obj)
                if force or _stale(obj, src):
                    jobs.append([cc, *ARCH, *FLAGS, *vflags, f"-DJGDPA_HEAD_DIM={d}", "-c", src, "-o", obj])
    return jobs, objs


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles every object that is out of date (in parallel) and links both
    libraries; returns the product library's path."""
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    jobs, objs = _compile_jobs(cc, force)
    if jobs:
        workers = max(1, min(len(jobs), os.cpu_count() or 1))
        with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
        for cmd, r in zip(jobs, results):
            if verbose and r.stderr:
                sys.stderr.write(r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    for v in VARIANTS:
        out = lib_path(v)
        if force or jobs or not os.path.exists(out):
            tmp = out + f".tmp{os.getpid()}"
            r = subprocess.run([cc, *ARCH, "-shared", "-cudart", "static", *objs[v], "-o", tmp],
                               capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, out)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

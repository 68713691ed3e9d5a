"""Builds libkvq.so in-tree with nvcc for sm_103a (no torch extension machinery).

    python -m int4_quantized_paged_gb300.build
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
OUT = os.path.join(PKG, "libkvq.so")
BUILD = os.path.join(PKG, "_build")
SOURCES = ["api.cu", "write.cu", "decode.cu", "prefill.cu", "prefill_ws.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libkvq")


def _headers_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    paths.append(os.path.join(ROOT, "include", "kvq.h"))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, extra: list | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    hdr = _headers_mtime()
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), hdr):
            jobs.append([cc, *ARCH, *FLAGS, *(extra or []), "-c", s, "-o", o])
    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr
    with cf.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        for msg in ex.map(run, jobs):
            if verbose and msg:
                sys.stderr.write(msg)
    if jobs or not os.path.exists(OUT):
        tmp = OUT + f".tmp{os.getpid()}"
        run([cc, *ARCH, "-shared", *objs, "-o", tmp])
        os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    # --force rebuilds every object; --ptxas-v prints register and spill
    # counts; -DNAME=VALUE arguments set the kernels' build-time knobs
    extra = [a for a in sys.argv[1:] if a.startswith("-D")]
    if "--ptxas-v" in sys.argv:
        extra += ["-Xptxas", "-v"]
    print(build(force="--force" in sys.argv or bool(extra), verbose=True, extra=extra or None))

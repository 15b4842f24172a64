"""Build libnvfp4fc2.so in-tree for sm_103a (nvcc, no cmake).

Steps: generate the BF16 silu table header, compile each .cu in parallel
with ``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3`` (IEEE
division and square root, no flush-to-zero, no fast math), link a shared
library with the CUDA runtime linked statically.  Output:
``diffusion_transformer_mlp_gb300/_build/libnvfp4fc2.so``.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
GEN = os.path.join(BUILD, "gen")
LIB = os.path.join(BUILD, "libnvfp4fc2.so")
SOURCES = ["api.cu", "quant.cu", "gemm.cu", "mma_peak.cu", "tc_read.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-ftz=false", "-prec-div=true",
                     "-prec-sqrt=true", "-fmad=true", "-Xptxas", "-v"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _newer(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(GEN, exist_ok=True)
    table = os.path.join(GEN, "silu_table_full.inc")
    gen = os.path.join(CSRC, "gen_silu_table.py")
    if force or _newer(table, [gen]):
        subprocess.check_call([sys.executable, gen, table])
    deps = _headers() + [table]
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _newer(o, [s] + deps):
            cmd = [nvcc()] + NVCC_FLAGS + ["-I", INCLUDE, "-I", CSRC, "-I", GEN, "-c", s, "-o", o]
            jobs.append((src, cmd))

    def run(job):
        src, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        for src, r in ex.map(run, jobs):
            log = r.stdout + r.stderr
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{log}")
            with open(os.path.join(BUILD, src + ".ptxas.txt"), "w") as f:
                f.write(log)
            if verbose:
                print(log)
    if force or jobs or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))

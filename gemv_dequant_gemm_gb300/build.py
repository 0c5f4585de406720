"""Build libqmm.so in-tree with nvcc for sm_103a (GB300).

Each csrc/*.cu is compiled to an object in parallel, then linked into
gemv_dequant_gemm_gb300/libqmm.so (CUDA runtime linked statically).
ptxas resource usage (-Xptxas -v) is written to _build/ptxas_<file>.log.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libqmm.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    for src in _sources():
        obj = os.path.join(BUILD, src[:-3] + ".o")
        log = open(os.path.join(BUILD, f"ptxas_{src[:-3]}.log"), "w")
        cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, obj, log, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT)))
    objs, failed = [], []
    for src, obj, log, p in procs:
        p.wait()
        log.close()
        objs.append(obj)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        msgs = []
        for src in failed:
            with open(os.path.join(BUILD, f"ptxas_{src[:-3]}.log")) as f:
                msgs.append(f"--- {src} ---\n" + f.read()[-6000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)

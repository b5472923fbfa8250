"""Build the in-tree CUDA libraries for sm_103a with nvcc (no cmake).

libzs.so        the C ABI of include/zs.h (package csrc/)
libzs_synth.so  the synthetic-input generator (synth/csrc/)

Translation units compile in parallel; a library is rebuilt only when one
of its sources or headers is newer than it.  ptxas register / spill reports
go to <package>/_build/ptxas_<unit>.log.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
SYNTH = os.path.join(ROOT, "synth")
BUILD = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "-prec-div=true", "-prec-sqrt=true", "-ftz=false"]

LIBZS = os.path.join(PKG, "libzs.so")
LIBSYNTH = os.path.join(SYNTH, "libzs_synth.so")


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzs")
    return cand


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run_parallel(jobs):
    procs = []
    for cmd, log in jobs:
        f = open(log, "w")
        procs.append((subprocess.Popen(cmd, stdout=f, stderr=subprocess.STDOUT), f, cmd, log))
    failed = []
    for p, f, cmd, log in procs:
        p.wait()
        f.close()
        if p.returncode != 0:
            failed.append((cmd, log))
    if failed:
        msgs = []
        for cmd, log in failed:
            with open(log) as f:
                msgs.append(" ".join(cmd) + "\n" + f.read()[-4000:])
        raise RuntimeError("build failed:\n" + "\n".join(msgs))


def _build_lib(name, target, cu_srcs, cpp_srcs, incs, deps, force=False):
    if not force and not _newer(target, deps):
        return False
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    inc = [f"-I{d}" for d in incs]
    jobs, objs = [], []
    for src in cu_srcs:
        stem = os.path.splitext(os.path.basename(src))[0]
        obj = os.path.join(BUILD, f"{name}_{stem}.o")
        jobs.append(([nvcc, *ARCH, *NVCC_FLAGS, *inc, "-c", src, "-o", obj],
                     os.path.join(BUILD, f"ptxas_{name}_{stem}.log")))
        objs.append(obj)
    for src in cpp_srcs:
        stem = os.path.splitext(os.path.basename(src))[0]
        obj = os.path.join(BUILD, f"{name}_{stem}.o")
        jobs.append((["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", *inc,
                      f"-I{os.path.join(os.path.dirname(nvcc), '..', 'include')}",
                      "-c", src, "-o", obj],
                     os.path.join(BUILD, f"gcc_{name}_{stem}.log")))
        objs.append(obj)
    _run_parallel(jobs)
    tmp = target + ".tmp"
    _run_parallel([([nvcc, *ARCH, "-shared", "-o", tmp, *objs],
                    os.path.join(BUILD, f"link_{name}.log"))])
    os.replace(tmp, target)
    return True


def build(force: bool = False, verbose: bool = False) -> None:
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hdrs.append(os.path.join(INCLUDE, "zs.h"))
    cu = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith(".cu")]
    cpp = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith(".cpp")]
    b1 = _build_lib("zs", LIBZS, cu, cpp, [INCLUDE, CSRC], cu + cpp + hdrs, force)
    scsrc = os.path.join(SYNTH, "csrc")
    scu = [os.path.join(scsrc, f) for f in sorted(os.listdir(scsrc)) if f.endswith(".cu")]
    b2 = _build_lib("synth", LIBSYNTH, scu, [], [scsrc], scu, force)
    if verbose:
        print(f"libzs: {'built' if b1 else 'up to date'}; libzs_synth: {'built' if b2 else 'up to date'}")


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)

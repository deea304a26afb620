"""Build libexl3.so in-tree with nvcc for sm_103a.

Each translation unit compiles to an object in parallel (the GEMM is compiled
once per trellis width), then nvcc links the shared library next to this file.
No CMake, no torch extension machinery: the library exposes a plain C ABI.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libexl3.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def units():
    """(source, object, extra flags) for every translation unit."""
    out = []
    for name in ("exl3_api.cu", "exl3_transform.cu", "exl3_kernels_misc.cu", "exl3_tc_host.cu", "exl3_noalloc.cu"):
        out.append((name, name.replace(".cu", ".o"), []))
    for b in range(1, 9):
        out.append(("exl3_gemm_tc_inst.cu", f"exl3_gemm_tc_b{b}.o", [f"-DEXL3_INST_BITS={b}"]))
    return out


def _flags():
    f = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"] + ARCH
    if os.environ.get("EXL3_PTXAS_VERBOSE"):
        f += ["-Xptxas", "-v"]
    return f


def _newer(obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return False
    t = os.path.getmtime(obj)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    headers.append(os.path.join(os.path.dirname(PKG), "include", "exl3.h"))
    jobs = []
    objs = []
    for src, obj, extra in units():
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, obj)
        objs.append(o)
        if force or not _newer(o, [s] + headers):
            jobs.append([cc, *_flags(), *extra, "-c", s, "-o", o])

    def run(cmd):
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p

    failed = []
    if jobs:
        workers = max(1, min(len(jobs), os.cpu_count() or 4))
        with ThreadPoolExecutor(workers) as ex:
            for cmd, p in ex.map(run, jobs):
                if verbose or p.returncode:
                    sys.stderr.write(" ".join(cmd[-3:]) + "\n" + p.stdout + p.stderr)
                if p.returncode:
                    failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if force or jobs or not _newer(LIB, objs):
        cmd = [cc, "-shared", *ARCH, "-o", LIB, *objs, "-cudart", "static"]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode:
            raise RuntimeError("link failed:\n" + p.stdout + p.stderr)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))

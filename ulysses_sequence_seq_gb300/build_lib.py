"""Build ``libusp.so`` (the C-ABI CUDA library) in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library with the CUDA runtime linked statically. No CMake, no torch
extension machinery: the library exports plain ``extern "C"`` symbols.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libusp.so")
SOURCES = ["relayout.cu", "sched.cu", "attn_fwd.cu", "attn_bwd.cu", "usp_api.cu", "noalloc.cu", "sp_loss.cu", "a2a.cu", "ring.cu"]

# Kernels that rebalance registers between warpgroups with setmaxnreg: the increase waits
# until the decreases have returned enough of the registers the CTA was launched with, so
# the launch allocation (registers per thread reported by ptxas) must be at least this
# many, or the kernel would never get past that point. Checked on every build.
MIN_LAUNCH_REGS = {"attn_fwd_kernel": 168}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libusp")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh"))]
    files.append(os.path.join(INCLUDE, "usp.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def check_launch_registers(ptxas_log: str) -> None:
    """Fail the build when a setmaxnreg kernel was allocated fewer launch registers than its split needs."""
    current = None
    seen = {}
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            for name in MIN_LAUNCH_REGS:
                if name in current:
                    seen.setdefault(name, []).append(int(m.group(1)))
    for name, need in MIN_LAUNCH_REGS.items():
        got = seen.get(name)
        if not got:
            raise RuntimeError(f"ptxas report for {name} not found; cannot check its register split")
        if min(got) < need:
            raise RuntimeError(f"{name} launched with {min(got)} registers per thread; its setmaxnreg "
                               f"split needs {need}")


def build(force: bool = False, verbose: bool = False, defines=()) -> str:
    """Compile every translation unit and link libusp.so. `defines` adds preprocessor
    symbols (e.g. USP_TIMELINE for the backward's optional clock64 timeline)."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC,
                     "-Xptxas", "-v"] + ["-D" + d for d in defines]

    def compile_one(src):
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + common
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, err in results:
            if err:
                print(err)
    check_launch_registers("\n".join(err for _, err in results))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", "-o", tmp] + [o for o, _ in results] + ARCH + ["-cudart=static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))

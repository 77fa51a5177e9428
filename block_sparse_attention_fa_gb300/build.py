"""Build the C-ABI shared library ``_lib/libfa_gb300.so`` from ``csrc/``.

Each CUDA translation unit is compiled for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``) in parallel, then linked with
the shared CUDA runtime.  Rebuilds only when a source is newer than the
library.  Usable as ``python -m block_sparse_attention_fa_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libfa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _cuda_home(nv: str) -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nv)))


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


# Kernels that move registers between warpgroups with setmaxnreg: the shares
# they hand out add up to a fixed per-thread launch count, so the compiled
# kernel must be launched with exactly that many registers (a smaller launch
# allocation would leave a setmaxnreg.inc waiting for registers forever).
LAUNCH_REGISTERS = {"fwd_bf16.cu": ("fwd_bf16_kernel", 168)}


def check_launch_registers(src: str, ptxas_log: str) -> None:
    if src not in LAUNCH_REGISTERS:
        return
    kernel, want = LAUNCH_REGISTERS[src]
    got = []
    current = None
    for line in ptxas_log.splitlines():
        if "Compiling entry function" in line:
            current = line
        elif "Used" in line and "registers" in line and current and kernel in current:
            got.append(int(line.split("Used")[1].split("registers")[0]))
    if not got or any(g != want for g in got):
        raise RuntimeError(f"{src}: {kernel} must launch with {want} registers per thread, ptxas reports {got}")


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nv = nvcc()
    os.makedirs(LIBDIR, exist_ok=True)
    objdir = os.path.join(LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                    "-I", CSRC, "-I", INCLUDE]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        extra = ["-Xptxas", "-v"] if os.path.basename(src) in LAUNCH_REGISTERS and not ptxas_verbose else []
        cmd = [nv] + flags + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        check_launch_registers(os.path.basename(src), r.stderr)
        if verbose or ptxas_verbose:
            sys.stderr.write(r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    libdir = os.path.join(_cuda_home(nv), "lib64")
    cmd = [nv] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "shared", "-Xlinker", f"-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))

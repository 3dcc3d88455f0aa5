"""Build ``libtfl.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

The translation units in ``csrc/`` are compiled in parallel, then linked into
``attention_qkv_gemm_gb300/libtfl.so``.  Objects go to ``_build/`` next to
this file.  A rebuild happens only when a source or header is newer than the
library (or ``force=True``).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtfl.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]
SOURCES = ["gemm.cu", "attention.cu", "attention_bwd.cu", "postchain.cu", "stack.cu", "rows.cu", "api.cu"]

# The attention kernels that run two CTAs of 256 threads per SM move registers from their first
# warpgroup to the second with setmaxnreg (64 and 192 a thread).  That balances only when the
# kernel launches with exactly 128 registers a thread: launched with fewer, setmaxnreg.inc would
# wait on the GPU for registers that never come free.  ptxas reports the launch count of every
# entry function; a build that does not give these kernels exactly 128 is refused.
SETMAXNREG_LAUNCH_REGS = {
    "_ZN3tfl11attn_kernelILi32EEEv": 128,  # attn_kernel<32>
    "_ZN3tfl11attn_kernelILi64EEEv": 128,  # attn_kernel<64>
}
PTXAS_INFO_SOURCES = {"attention.cu"}


def launch_registers(ptxas_log: str) -> dict:
    """Registers a thread at launch of each entry function in a ``-Xptxas -v`` log."""
    regs, cur = {}, None
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and cur is not None:
            regs[cur] = int(m.group(1))
            cur = None
    return regs


def check_launch_registers(ptxas_log: str, required: dict = SETMAXNREG_LAUNCH_REGS) -> None:
    """Raise unless every kernel whose mangled name starts with a key of ``required`` was
    compiled, and launches with exactly the given registers a thread."""
    regs = launch_registers(ptxas_log)
    for prefix, want in required.items():
        got = {k: v for k, v in regs.items() if k.startswith(prefix)}
        if not got:
            raise RuntimeError(f"ptxas reported no register count for {prefix}")
        for k, v in got.items():
            if v != want:
                raise RuntimeError(f"{k} launches with {v} registers a thread; its setmaxnreg split "
                                   f"needs exactly {want}")


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin directory on PATH)")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "tfl.h"))
    return files


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link; returns the library path."""
    if not force and not ptxas_info and not needs_build():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        info = extra if extra or src not in PTXAS_INFO_SOURCES else ["-Xptxas", "-v"]
        cmd = [nvcc, *ARCH, *FLAGS, *info, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    logs = []
    for src, _, r in results:
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if src in PTXAS_INFO_SOURCES:
            check_launch_registers(r.stdout + r.stderr)
        if verbose or ptxas_info:
            logs.append(f"== {src}\n{r.stdout}{r.stderr}")
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if logs:
        sys.stdout.write("\n".join(logs))
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)

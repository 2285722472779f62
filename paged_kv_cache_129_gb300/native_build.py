"""Build the CUDA library ``_build/libpagedkv.so`` for sm_103a with nvcc.

Each translation unit is compiled in parallel; the host pool is plain C++.
The CUDA runtime is linked statically, so the library loads without a GPU
(for the export checks) and shares the driver's primary context with PyTorch.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpagedkv.so")

CUDA_SOURCES = ["capi.cu", "kv_ops.cu", "decode_f32.cu", "decode_f16.cu", "decode_bf16.cu", "decode_fp8.cu",
                "decode_static_scratch.cu"]
CXX_SOURCES = ["block_pool.cpp", "stepper.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _deps() -> list:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(BUILD, ".flags"))
    files.append(os.path.join(INCLUDE, "pa.h"))
    files.append(os.path.abspath(__file__))
    return files


def _flags_file_current() -> None:
    """Record the extra flags; a change of flags makes the library stale."""
    os.makedirs(BUILD, exist_ok=True)
    path = os.path.join(BUILD, ".flags")
    flags = os.environ.get("PA_NVCC_EXTRA", "")
    if not os.path.exists(path) or open(path).read() != flags:
        with open(path, "w") as f:
            f.write(flags)


def up_to_date() -> bool:
    _flags_file_current()
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _run(cmd: list) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int = 0) -> str:
    """Compile every translation unit and link the shared library; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ["-std=c++17", "-O3", "-I", INCLUDE, "-I", CSRC, "-Xcompiler", "-fPIC"]
    # Optional extra nvcc flags for tuning builds (e.g. -DPA_LEAN_RING_KB=96).
    common += os.environ.get("PA_NVCC_EXTRA", "").split()
    cmds, objs = [], []
    for src in CUDA_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        flags = ARCH + ["-lineinfo", "--expt-relaxed-constexpr"] + (["-Xptxas", "-v"] if verbose_ptxas else [])
        cmds.append([cc, "-c", os.path.join(CSRC, src), "-o", obj] + common + flags)
        objs.append(obj)
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        cmds.append([cc, "-c", "-x", "c++", os.path.join(CSRC, src), "-o", obj] + common)
        objs.append(obj)
    workers = jobs or min(len(cmds), os.cpu_count() or 1)
    with ThreadPoolExecutor(workers) as pool:
        list(pool.map(_run, cmds))
    tmp = LIB + f".tmp{os.getpid()}"
    _run([cc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static", "-Xcompiler", "-fPIC"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-v", action="store_true", help="print register/spill/shared-memory usage")
    args = ap.parse_args()
    print(build(force=args.force or args.ptxas_v, verbose_ptxas=args.ptxas_v))

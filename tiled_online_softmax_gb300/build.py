"""Build libfa.so (the sm_103a attention kernels and their C interface) in place with nvcc, and
libfa_debug.so, the same library with every global store bounds-checked (FA_DEBUG_BOUNDS)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
LIB = PKG / "libfa.so"
DEBUG_LIB = PKG / "libfa_debug.so"
SOURCES = [CSRC / "fa_api.cu"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-Xcompiler", "-fPIC", "-shared",
    "-Xptxas", "-v",
    f"-I{ROOT / 'include'}", f"-I{CSRC}",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found")


def build(verbose: bool = False) -> Path:
    """Compile every CUDA source into libfa.so and libfa_debug.so next to this file (two nvcc
    processes in parallel); return the path of libfa.so."""
    jobs = [(LIB, [], PKG / "build.log"), (DEBUG_LIB, ["-DFA_DEBUG_BOUNDS"], PKG / "build_debug.log")]
    procs = []
    for out, extra, log in jobs:
        tmp = out.with_suffix(".so.tmp")
        cmd = [nvcc(), *NVCC_FLAGS, *extra, "-o", str(tmp), *map(str, SOURCES)]
        procs.append((out, tmp, log, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                            stderr=subprocess.PIPE, text=True)))
    failed = []
    for out, tmp, log, cmd, proc in procs:
        stdout, stderr = proc.communicate()
        log.write_text(" ".join(cmd) + "\n" + stdout + stderr)
        if proc.returncode != 0:
            sys.stderr.write(stdout + stderr)
            failed.append(f"{out.name}: nvcc failed ({proc.returncode}); see {log}")
            continue
        if verbose:
            sys.stderr.write(stdout + stderr)
        tmp.replace(out)
    if failed:
        raise RuntimeError("; ".join(failed))
    return LIB


if __name__ == "__main__":
    build(verbose=True)
    print(LIB)

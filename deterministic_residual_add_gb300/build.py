"""Build libdradd.so in-tree with nvcc for sm_103a.

Each .cu translation unit is compiled in parallel, then linked into a shared
library next to this file.  `python -m deterministic_residual_add_gb300.build`
builds it from the command line.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import threading
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIB = PKG / "libdradd.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# No fast math: IEEE division and square root, no flush to zero, and no
# contraction of a multiply and an add into one fused operation.
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-fmad=false",
              "-prec-div=true", "-prec-sqrt=true", "-ftz=false", "-Xptxas", "-v"]

_lock = threading.Lock()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdradd")


def _sources():
    return sorted(CSRC.glob("*.cu"))


def _deps():
    return _sources() + sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + sorted(INCLUDE.glob("*.h"))


def stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    return any(p.stat().st_mtime > t for p in _deps())


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile and link libdradd.so if it is missing or older than a source."""
    with _lock:
        if not force and not stale():
            return LIB
        BUILD.mkdir(exist_ok=True)
        cc = nvcc()

        def compile_one(src: Path) -> Path:
            obj = BUILD / (src.stem + ".o")
            cmd = [cc, *ARCH, *NVCC_FLAGS, "-I", str(INCLUDE), "-I", str(CSRC), "-c", str(src),
                   "-o", str(obj)]
            r = subprocess.run(cmd, capture_output=True, text=True)
            (BUILD / (src.stem + ".ptxas.txt")).write_text(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src.name}:\n{r.stdout}\n{r.stderr}")
            return obj

        srcs = _sources()
        with ThreadPoolExecutor(len(srcs)) as ex:
            objs = list(ex.map(compile_one, srcs))
        tmp = LIB.with_suffix(f".so.tmp{os.getpid()}")
        cmd = [cc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
        if verbose:
            for f in sorted(BUILD.glob("*.ptxas.txt")):
                print(f.read_text())
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)

"""In-tree build of the CUDA library (sm_103a) and, for the test suite, the
CPU oracle.

``build_library()`` compiles every ``csrc/*.cu`` translation unit in parallel
with nvcc for ``sm_103a`` and links ``libbd.so`` next to this file (static
CUDA runtime, so the library needs only the driver at run time).
``build_oracle()`` compiles ``oracle/bd_oracle.c`` with gcc; building the
checker does not load or run it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libbd.so")
OBJ = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbd.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False) -> str:
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    heads = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                   glob.glob(os.path.join(ROOT, "include", "*.h")))
    if not force and not _stale(LIB, srcs + heads):
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    nv = nvcc()

    def compile_one(src):
        obj = os.path.join(OBJ, os.path.basename(src) + ".o")
        cmd = [nv, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, err in results:
            print(err)
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nv, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def build_oracle(force: bool = False) -> str:
    src = os.path.join(ROOT, "oracle", "bd_oracle.c")
    out = os.path.join(ROOT, "oracle", "liboracle.so")
    if force or _stale(out, [src]):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                               src, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    build_library(force="--force" in sys.argv, verbose="-v" in sys.argv)
    build_oracle(force="--force" in sys.argv)
    print(LIB)

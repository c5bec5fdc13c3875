"""Build libkq.so (the sm_103a CUDA library) in-tree with nvcc.

    python -m quant_quantized_matvec_gb300.build [--force]

The library lands in quant_quantized_matvec_gb300/lib/libkq.so (git-ignored).
A build is skipped when the library is newer than every source and header.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "lib", "libkq.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__])


def nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _inputs())


def _compile(args):
    src, obj, verbose = args
    cmd = [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, r.returncode, r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every .cu under csrc/ in parallel, then link libkq.so."""
    if not force and not is_stale():
        return LIB
    from concurrent.futures import ThreadPoolExecutor
    objdir = os.path.join(PKG, "lib", "obj")
    os.makedirs(objdir, exist_ok=True)
    jobs = [(src, os.path.join(objdir, os.path.basename(src) + ".o"), verbose)
            for src in sources()]
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(_compile, jobs))
    failed = [(s, out) for s, rc, out in results if rc != 0]
    for s, rc, out in results:
        if verbose or rc != 0:
            print(out, end="", flush=True)
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(s for s, _ in failed))
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), ARCH, "-shared", "-o", tmp] + [j[1] for j in jobs],
                   check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

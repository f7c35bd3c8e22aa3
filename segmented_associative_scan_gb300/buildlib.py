"""Build librlca.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own nvcc process, in parallel (the reverse
estimators once per estimator and input format, the forward scans once per format), then
the objects are linked into one shared library with the CUDA runtime linked statically.
Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librlca.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librlca")
    return path


# Sources compiled more than once, one object per set of defines: each reverse
# estimator in each input format, and the forward scans in each format.
VARIANTS = {
    "reverse_unit.cu": [{"RLCA_UNIT_EST": e, "RLCA_UNIT_FMT": f}
                        for e in range(5) for f in range(3)],
    "forward_unit.cu": [{"RLCA_UNIT_FMT": f} for f in range(3)],
}


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def units() -> list[tuple[str, dict]]:
    """(source, defines) for every object of the library."""
    out = []
    for src in sources():
        for defs in VARIANTS.get(os.path.basename(src), [{}]):
            out.append((src, defs))
    return out


def _deps() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and not ptxas_info and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(unit):
        src, defs = unit
        tag = "".join(f".{v}" for v in defs.values())
        obj = os.path.join(BUILD, os.path.basename(src) + tag + ".o")
        dflags = [f"-D{k}={v}" for k, v in defs.items()]
        cmd = [cc, *ARCH, *FLAGS, *extra, *dflags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    # Longest first: the reverse units dominate the build.
    todo = sorted(units(), key=lambda u: os.path.basename(u[0]) != "reverse_unit.cu")
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, todo))
    if verbose or ptxas_info:
        for _, log in results:
            if log:
                sys.stderr.write(log)
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))

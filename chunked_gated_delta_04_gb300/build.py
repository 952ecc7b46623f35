"""Build libgdr.so in-tree: every csrc/*.cu compiled for sm_103a only, in parallel, then linked.

    python -m chunked_gated_delta_04_gb300.build [--force] [--debug]

nvcc flags: -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -lineinfo, no fast-math.
Each device pass checks __CUDA_ARCH_FEAT_SM103_ALL and fails if the gencode was lost.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libgdr.so")
BUILD_DIR = os.path.join(PKG, "_build")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdr.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))) + [
        os.path.join(INCLUDE, "gdr.h")]


FLAGS_STAMP = LIB + ".flags"  # the flags the library was built with (a rebuild when they change)


def _flags(debug: bool = False) -> list:
    flags = GENCODE + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                       "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]
    if debug:
        flags += ["-DGDR_DEBUG_DELAY=1"]
    return flags + os.environ.get("GDR_NVCC_EXTRA", "").split()


def up_to_date(debug: bool = False) -> bool:
    if not os.path.exists(LIB) or not os.path.exists(FLAGS_STAMP):
        return False
    with open(FLAGS_STAMP) as f:
        if f.read() != " ".join(_flags(debug)):
            return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, debug: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date(debug):
        return LIB
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    flags = _flags(debug)
    stamp = " ".join(flags)
    if verbose:
        flags = flags + ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose:
        for _, err in results:
            print(err)
    objs = [o for o, _ in results]
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc] + GENCODE + ["-shared", "-o", tmp] + objs + ["-lcudart_static", "-ldl",
                                                                "-lrt", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(FLAGS_STAMP, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--debug", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, debug=args.debug, verbose=args.verbose))

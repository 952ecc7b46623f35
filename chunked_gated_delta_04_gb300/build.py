"""Build libgdr.so in-tree: every csrc/*.cu compiled for sm_103a only, in parallel, then linked.

    python -m chunked_gated_delta_04_gb300.build [--force] [--delay]

--delay builds the delay-injection variant libgdr_delay.so instead (-DGDR_DEBUG_DELAY: one role
at each cross-role hand-off sleeps a short bounded time; see csrc/gdr_instrument.cuh), which the
tests compare bit for bit with libgdr.so.

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
DELAY_LIB = os.path.join(PKG, "libgdr_delay.so")
DELAY_BUILD_DIR = os.path.join(PKG, "_build_delay")
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


def _target(delay: bool):
    """(library path, object directory, flags stamp) of the normal or the delay-injection build."""
    lib = DELAY_LIB if delay else LIB
    return lib, (DELAY_BUILD_DIR if delay else BUILD_DIR), lib + ".flags"


def _flags(delay: bool = False) -> list:
    flags = GENCODE + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                       "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]
    if delay:
        flags += ["-DGDR_DEBUG_DELAY=1"]
    return flags + os.environ.get("GDR_NVCC_EXTRA", "").split()


def up_to_date(delay: bool = False) -> bool:
    lib, _, stamp = _target(delay)
    if not os.path.exists(lib) or not os.path.exists(stamp):
        return False
    with open(stamp) as f:
        if f.read() != " ".join(_flags(delay)):
            return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, delay: bool = False, verbose: bool = False) -> str:
    """Builds libgdr.so (or, with delay, libgdr_delay.so) unless it is up to date; returns its path."""
    lib, build_dir, stamp_path = _target(delay)
    if not force and up_to_date(delay):
        return lib
    nvcc = nvcc_path()
    os.makedirs(build_dir, exist_ok=True)
    flags = _flags(delay)
    stamp = " ".join(flags)
    if verbose:
        flags = flags + ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
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
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + GENCODE + ["-shared", "-o", tmp] + objs + ["-lcudart_static", "-ldl",
                                                                "-lrt", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--delay", action="store_true", help="build the delay-injection variant libgdr_delay.so")
    ap.add_argument("-v", "--verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, delay=args.delay, verbose=args.verbose))

"""Build libzeroshard.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ is compiled in parallel to an object file,
then linked into ``_build/libzeroshard.so`` against the shared CUDA runtime
(the one the PyTorch process has already loaded).  ptxas resource usage of
every kernel is kept in ``_build/ptxas.log``.

The same sources built with -DZERO_DEBUG give ``_build/debug/
libzeroshard_debug.so``: every kernel checks its access indices and
alignments and records violations instead of faulting (zero_debug_errors).
The binding loads it instead of the release library when the environment
sets ZERO_SHARD_DEBUG=1.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libzeroshard.so")
DEBUG_BUILD = os.path.join(BUILD, "debug")
DEBUG_LIB = os.path.join(DEBUG_BUILD, "libzeroshard_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-ffp-contract=off", "-Xptxas", "-v",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzeroshard")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link the release library (and, with debug=True, the debug one
    too, in the same parallel pass); returns the release library's path."""
    variants = [(BUILD, LIB, [])] + ([(DEBUG_BUILD, DEBUG_LIB, ["-DZERO_DEBUG"])] if debug else [])
    variants = [v for v in variants if force or _stale(v[1])]
    if not variants:
        return LIB
    cc = nvcc()
    procs = []
    for out_dir, _, extra in variants:
        os.makedirs(out_dir, exist_ok=True)
        for src in sources():
            obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
            cmd = [cc] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
            procs.append((out_dir, src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                                         text=True)))
    logs = {v[0]: [] for v in variants}
    failed = []
    for out_dir, src, p in procs:
        out, _ = p.communicate()
        logs[out_dir].append(f"==== {os.path.basename(src)}\n{out}")
        if p.returncode != 0:
            failed.append(src)
    for out_dir, lines in logs.items():
        with open(os.path.join(out_dir, "ptxas.log"), "w") as f:
            f.write("\n".join(lines))
    if failed:
        sys.stderr.write("\n".join(sum(logs.values(), [])))
        raise RuntimeError(f"nvcc failed on {', '.join(os.path.basename(s) for s in failed)}")
    for out_dir, lib, _ in variants:
        objs = [os.path.join(out_dir, os.path.basename(src)[:-3] + ".o") for src in sources()]
        tmp = lib + f".tmp{os.getpid()}"
        link = [cc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + \
            ["-Xlinker", "-rpath,/usr/local/cuda/lib64"]
        subprocess.run(link, check=True)
        os.replace(tmp, lib)
    if verbose:
        print("\n".join(sum(logs.values(), [])))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))

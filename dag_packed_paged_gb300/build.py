"""Build libtreeattn.so in-tree with nvcc for sm_103a (no CMake; objects compiled in parallel)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libtreeattn.so")
# The same library compiled with -DTA_DEBUG: every kernel checks its page-table lookups, TMA
# pool rows and output rows on the device and reports a failed check through the plan's status
# word (tree_attn_check: TA_ERR_DEVICE_BOUNDS) instead of touching memory out of range.  Loaded
# instead of LIB when TREEATTN_DEBUG=1.
LIB_DEBUG = os.path.join(BUILD, "libtreeattn_debug.so")
SOURCES = ["plan.cpp", "ingest.cpp", "place.cpp", "api.cu", "fwd.cu", "fwd_pair.cu", "bwd.cu", "rope.cu", "logprob.cu", "noalloc.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtreeattn")
    return cand


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "treeattn.h"))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    out = LIB_DEBUG if debug else LIB
    if not force and os.path.exists(out) and os.path.getmtime(out) >= _deps():
        return out
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                     "--expt-relaxed-constexpr"] + (["-DTA_DEBUG"] if debug else [])
    tag = f"{os.getpid()}{'d' if debug else ''}"

    def compile_one(src):
        obj = os.path.join(BUILD, src + f".{tag}.o")
        cmd = [nvcc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + f".{tag}.tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
        "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, out)
    for o in objs:
        os.remove(o)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))

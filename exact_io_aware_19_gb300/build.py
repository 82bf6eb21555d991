"""Build libattn.so in-tree: every translation unit of csrc/ for sm_103a, in parallel.

    python -m exact_io_aware_19_gb300.build [--force] [--verbose]

Output: exact_io_aware_19_gb300/_build/libattn.so (git-ignored). The CUDA runtime is
linked statically, so the library only needs the NVIDIA driver at run time.
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-DNDEBUG",
              "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(INCLUDE, "attn.h"), __file__]


STAMP = os.path.join(BUILD, "flags.txt")


def _defines():
    """Tuning defines taken from the environment: EX19_POLY_PAIRS (pairs of every 8
    softmax columns whose exp2 runs on the FMA-pipe polynomial; default 0),
    EX19_SEPARATE_P (d = 64 fp16 keeps P in its own TMEM columns; default 1),
    EX19_SOFTMAX_F2 (paired fp32 FMA / adds in the softmax; default 1),
    EX19_MAX3 (3-input max instruction in the row max; default 1),
    EX19_SUSPEND_NS (sleep hint of the mbarrier polls in ns; default 1e6, 0 = none),
    EX19_TRACE (CTA 0 records a clock64 timeline of its first unit in the workspace; default 0),
    EX19_ONEPASS (the softmax reads S from TMEM once instead of twice; default 1),
    EX19_SPIN (bounded waits spin on mbarrier.test_wait instead of try_wait; default 0),
    EX19_EXP_F16X2 (fp16: packed fp16 exponentials, two per MUFU operation; default 1),
    EX19_PV_HALVES (separate P: P handed to the P·V MMAs in two 64-key halves; default 1)."""
    out = []
    for name in ("EX19_POLY_PAIRS", "EX19_SEPARATE_P", "EX19_SOFTMAX_F2", "EX19_MAX3",
                 "EX19_SUSPEND_NS",
                 "EX19_TRACE", "EX19_ONEPASS", "EX19_SPIN", "EX19_PV_HALVES",
                 "EX19_EXP_F16X2"):
        if os.environ.get(name):
            out.append("-D%s=%d" % (name, int(os.environ[name])))
    return out


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return False
    if open(STAMP).read() != " ".join(_defines()):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libattn.so unless it is already newer than every input."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    extra = (["-Xptxas", "-v"] if verbose else []) + _defines()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as fh:
        fh.write(" ".join(_defines()))
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))

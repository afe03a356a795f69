"""Build libloco.so (the CUDA library behind include/loco.h) in-tree with nvcc.

    python -m bit_gradient_compression_gb300.build

Targets sm_103a only.  The translation units compile in parallel; the CUDA
runtime is linked statically so the library loads on a machine without a GPU
driver (calls then fail with LOCO_ERR_CUDA / an argument error).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libloco.so")

SOURCES = ["abi.cu", "compress.cu", "decode_reduce.cu", "adam.cu", "sgd.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: no multiply-add contraction anywhere; every fp32 product and sum
# in the kernels is its own rounded operation, as the method's definition states.
# Hidden visibility: only the LOCO_API entry points of include/loco.h are
# exported; the static CUDA runtime's symbols are kept out of the dynamic
# symbol table too (--exclude-libs), so nothing can be interposed between this
# library and other CUDA code in the same process.
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
                     "-I", INCLUDE, "-I", CSRC]
LINK_FLAGS = ARCH + ["-shared", "-cudart", "static", "-Xlinker", "--exclude-libs,ALL"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libloco")
    return path


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers():
    hs = [os.path.join(INCLUDE, "loco.h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str = LIB, build_dir: str = BUILD) -> str:
    """Compile the sources into build_dir and link them into out (default: in-tree libloco.so)."""
    os.makedirs(build_dir, exist_ok=True)
    headers = _headers()
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, *headers]):
            cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o]
            jobs.append(cmd)
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            futs = [ex.submit(subprocess.run, c, capture_output=True, text=True) for c in jobs]
            for c, f in zip(jobs, futs):
                r = f.result()
                if verbose or r.returncode != 0:
                    sys.stderr.write(" ".join(c) + "\n" + r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {c[-3]}")
    if force or jobs or _stale(out, objs):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc(), *LINK_FLAGS, "-o", tmp, *objs])
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

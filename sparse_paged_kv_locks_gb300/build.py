"""Build liblocks.so (sm_103a) in-tree with nvcc.

    python -m sparse_paged_kv_locks_gb300.build [--verbose]

Each .cu translation unit is compiled in parallel, then linked into
sparse_paged_kv_locks_gb300/lib/liblocks.so against the shared CUDA runtime
(the same libcudart the host process already uses).  `-Xptxas -v` output
(registers, spills, shared memory) is kept in lib/ptxas.log.
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
LIBDIR = os.path.join(PKG, "lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "liblocks.so")
SOURCES = ["api.cu", "build.cu", "score.cu", "select.cu", "decode.cu",
           "exact.cu", "variant.cu", "variant_b2.cu", "variant_b4.cu",
           "variant_b8.cu", "noalloc.cu", "decoder.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to "
                       "build liblocks.so")


def _compile(src: str) -> tuple:
    obj = os.path.join(OBJDIR, src.replace(".cu", ".o"))
    cmd = [nvcc(), *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xptxas", "-v",
           "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, "-c",
           os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr


def build(verbose: bool = False) -> str:
    os.makedirs(OBJDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    log = []
    for src, obj, rc, out in results:
        log.append(f"==== {src}\n{out}")
        if rc != 0:
            sys.stderr.write(out)
            raise RuntimeError(f"nvcc failed on {src}")
    objs = [obj for _, obj, _, _ in results]
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link of liblocks.so failed")
    os.replace(tmp, LIB)
    with open(os.path.join(LIBDIR, "ptxas.log"), "w") as f:
        f.write("\n".join(log))
    if verbose:
        print("\n".join(log))
    return LIB


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv))

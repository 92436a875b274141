"""Build the sm_103a shared library ``_build/libmla_decode_sm103.so`` with nvcc.

Each translation unit compiles in its own nvcc process (in parallel), then one
link step produces the library. Only ``-gencode arch=compute_103a,code=sm_103a``
is emitted: the kernels use tcgen05, TMA and cluster features of that target.
Run ``python -m paged_mla_decode_05_gb300.build`` from the repository root.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB_NAME = "libmla_decode_sm103.so"
LIB_PATH = os.path.join(BUILD, LIB_NAME)
SOURCES = ["mla_decode_sm103.cu", "mla_decode_rows_sm103.cu", "mla_combine_sm103.cu",
           "mla_no_alloc_sm103.cu", "mla_selftest_sm103.cu", "mla_sparse_sm103.cu", "mla_api.cpp"]
HEADERS = ["mla_internal.h", "ptx_sm103.cuh", "mla_decode_kernel.cuh"]
GENCODE = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "mla_decode.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if sources changed) and return the path of the shared library."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = [nvcc, GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        extra = ["-Xptxas", "-v"] if verbose and src.endswith(".cu") else []
        if src.endswith(".cu"):
            # No register may spill: the roles read tensor memory with
            # asynchronous loads whose destination registers must stay put
            # until the wait, which a spill between the two would break.
            extra += ["-Xptxas", "--warn-on-spills", "-Xptxas", "--warning-as-error"]
        cmds.append(common + extra + ["-c", os.path.join(CSRC, src), "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        for cmd, r in ex.map(run, cmds):
            if r.returncode != 0:
                raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
            if verbose and (r.stdout or r.stderr):
                sys.stderr.write(r.stdout + r.stderr)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, GENCODE, "-shared", "-o", tmp] + objs
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

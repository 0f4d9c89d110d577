"""In-tree build of the CUDA library (sm_103a only).

``python -m paged_mla_decode_09_gb300.build`` compiles
``csrc/mla_decode.cu`` (the decode), ``csrc/mla_kv_pack.cu`` (the cache
write), ``csrc/mla_sparse.cu`` (the top-k decode) and ``csrc/mla_cascade.cu``
(the shared-prefix cascade) with nvcc into ``libmla_decode.so`` next to this
file.  Four translation units, one ``-gencode``; a few seconds.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libmla_decode.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
SOURCES = [os.path.join(CSRC, f) for f in ("mla_decode.cu", "mla_kv_pack.cu", "mla_sparse.cu", "mla_cascade.cu")]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def depends():
    files = list(SOURCES)
    for d in (CSRC, INCLUDE):
        files += [os.path.join(d, f) for f in os.listdir(d) if f.endswith((".cuh", ".h"))]
    return files


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build the library")


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in depends())


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile the shared library in place; returns its path."""
    if not force and up_to_date():
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [
        nvcc_path(), "-shared", "-Xcompiler", "-fPIC", *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17",
        "-I", INCLUDE, "-I", CSRC, "-cudart", "shared", "-o", tmp, *SOURCES,
    ]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))

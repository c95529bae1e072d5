"""Build ``libbi.so`` (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each translation unit under ``csrc/`` is compiled by its own nvcc process
(in parallel), then linked with the static CUDA runtime into
``deterministic_invariant_bf16_gb300/libbi.so``.  The driver API is reached
through the runtime's entry-point query, so the library loads on hosts with
no GPU driver (the ABI tests need only ``dlopen``).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libbi.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(CSRC, "*.h")) +
            glob.glob(os.path.join(INCLUDE, "*.h")))


def source_hash(extra_flags=None) -> str:
    """sha256 over every source and header the library is built from and the
    compiler flags: the key that decides whether libbi.so is current (file
    times say nothing once a tree has been copied to another machine)."""
    h = hashlib.sha256()
    for path in sorted(_deps()):
        h.update(os.path.relpath(path, HERE).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS[:-2] + list(extra_flags or []))
             .encode())
    return h.hexdigest()


STAMP = LIB + ".sha256"


def _stale(extra_flags=None) -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return True
    with open(STAMP) as f:
        return f.read().strip() != source_hash(extra_flags)


def build(force: bool = False, verbose: bool = False,
          extra_flags=None) -> str:
    if not force and not _stale(extra_flags):
        return LIB
    key = source_hash(extra_flags)
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = ARCH + NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [cc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" %
                               (src, r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(key + "\n")
    return LIB


if __name__ == "__main__":
    force = "--force" in sys.argv
    flags = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None
    print(build(force=force or bool(flags), verbose=True, extra_flags=flags))

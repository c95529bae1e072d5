"""Compile the oracle's C core into ``oracle/_liboracle.so``.

TEST INFRASTRUCTURE ONLY: the oracle is the CPU checker of the GPU library.
Plain gcc, no architecture flags, so the same source builds on x86-64 and on
aarch64 hosts.  ``-ffp-contract=off`` keeps every fp32 multiply and add
separately rounded (gcc would otherwise fuse them into FMAs on aarch64).
"""
import hashlib
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "_liboracle.so")

CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
          "-shared", "-std=c11", "-Wall", "-Wextra", "-Wno-unused-parameter"]


STAMP = LIB + ".sha256"


def source_hash() -> str:
    """sha256 of the source and the flags: the library is rebuilt when it
    changes (file times do not survive a copy to another machine)."""
    h = hashlib.sha256(open(SRC, "rb").read())
    h.update(" ".join(CFLAGS).encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Build the shared library if it is missing or built from other
    sources or flags."""
    key = source_hash()
    if (not force and os.path.exists(LIB) and os.path.exists(STAMP)
            and open(STAMP).read().strip() == key):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(key + "\n")
    return LIB


if __name__ == "__main__":
    print(build(force=True))

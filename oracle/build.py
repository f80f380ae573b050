"""Compiles the fp64 oracle (gdr_oracle.c) into oracle/_lib/liboracle.so.

Test infrastructure only: the oracle is what the CUDA library is checked
against.  Plain gcc, no CUDA, portable C99 (builds the same on x86_64 and
aarch64 hosts).
"""
import os
import platform
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdr_oracle.c")
LIB_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIB_DIR, "liboracle.so")
STAMP = LIB + ".arch"  # the architecture the library was built on


def build(verbose: bool = False) -> str:
    os.makedirs(LIB_DIR, exist_ok=True)
    stamp_ok = os.path.exists(STAMP) and open(STAMP).read().strip() == platform.machine()
    if stamp_ok and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-O2", "-fPIC", "-shared",
           "-pthread", "-o", tmp, SRC, "-lm"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(platform.machine() + "\n")
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))

"""Build the fp64 CPU oracle (plain C) into oracle/libtw_oracle.so.

Test infrastructure only: the product library never loads what this builds.
Flags keep the arithmetic exactly as written (no fused multiply-add, no fast
math), so the x86 and Arm builds give the same fp64 bits.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "tw_oracle.c")
LIB = os.path.join(HERE, "libtw_oracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the oracle if the shared object is missing or stale; return its path."""
    srcs = [SRC, os.path.join(HERE, "tw_oracle.h")]
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(s) for s in srcs)):
        return LIB
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-shared", "-fPIC", "-o", LIB + ".tmp", SRC, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

"""Compiles the fp64 oracle (plain C) into oracle/liboracle.so with the host C compiler.

Test infrastructure: building the checker is not using it. Flags keep IEEE fp64
semantics identical on x86-64 and AArch64 (no FMA contraction, no fast-math).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp_oracle.c")
LIB_PATH = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC):
        return LIB_PATH
    cc = os.environ.get("CC", "gcc")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
           SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

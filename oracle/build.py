"""Compile the fp64 CPU oracle (plain C, gcc) into oracle/libattn_oracle.so.

Test infrastructure: the oracle is built so the tests, the smoke check and the
benchmark's CPU-baseline leg can call it; the product path never does.
Flags: -O2, no -ffast-math (plain IEEE exp/log and summation order), no
machine-specific flags, so it builds and behaves the same on x86_64 and aarch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
LIB = os.path.join(HERE, "libattn_oracle.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC),
                                            os.path.getmtime(os.path.join(HERE, "attn_oracle.h")))):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

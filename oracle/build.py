"""Compiles the C oracle into a shared library next to its source.

TEST INFRASTRUCTURE ONLY: the oracle is the checker the CUDA library is
compared against; building it is not using it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRCS = [os.path.join(HERE, "replayssm_oracle.c"), os.path.join(HERE, "gdn_commit_oracle.c")]
LIB = os.path.join(HERE, "_replayssm_oracle.so")

# -ffp-contract=off: no fused multiply-add, every fp32 step rounds on its own.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    deps = SRCS + [os.path.join(HERE, "replayssm_oracle.h"), os.path.join(HERE, "gdn_commit_oracle.h"),
                   os.path.abspath(__file__)]
    if not force and os.path.exists(LIB):
        if os.path.getmtime(LIB) >= max(os.path.getmtime(p) for p in deps):
            return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, *SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

"""Build the fp64 attention oracle, forward and gradients (test infrastructure),
with the host gcc.

Plain C11, IEEE binary64, ``-ffp-contract=off`` and no fast-math, so the
same source gives the same bits on x86-64 and AArch64 hosts.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRCS = [os.path.join(HERE, "attention_fp64.c"), os.path.join(HERE, "attention_bwd_fp64.c")]
LIB = os.path.join(HERE, "liboracle_fp64.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and all(os.path.getmtime(LIB) >= os.path.getmtime(src) for src in SRCS)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [os.environ.get("CC", "gcc"), "-O2", "-std=c11", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", "-pthread", "-o", tmp, *SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

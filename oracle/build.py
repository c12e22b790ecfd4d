"""Build step for the C oracle (test infrastructure): gcc -> liboracle.so.

Plain -O2 without fast-math, so float64 arithmetic keeps IEEE semantics and
the summation order written in attn_oracle.c.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
SO = os.path.join(HERE, "liboracle.so")


def build_oracle(force: bool = False) -> str:
    if (not force and os.path.exists(SO)
            and os.path.getmtime(SO) >= os.path.getmtime(SRC)):
        return SO
    tmp = SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-fno-fast-math", "-pthread", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, SO)
    return SO


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))

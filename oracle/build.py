"""Build the CPU oracle (``liboracle.so``) from ``moe_oracle.c`` with gcc.

Test infrastructure only: the oracle checks the GPU library, it is never
part of it.  The flags keep every binary32 operation separately rounded
(``-ffp-contract=off``, no fast-math), which is what makes the oracle a
plain definition that any conforming host reproduces bit for bit.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

BASE_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
              "-Wall", "-Wextra", "-Werror"]


def _compile(extra: list[str]) -> subprocess.CompletedProcess:
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *BASE_FLAGS, *extra, SRC, "-o", tmp, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode == 0:
        os.replace(tmp, LIB)
    elif os.path.exists(tmp):
        os.remove(tmp)
    return res


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    res = _compile(["-fopenmp"])
    if res.returncode != 0:
        # a host without OpenMP still gets the (single-threaded) oracle
        res2 = _compile(["-Wno-unknown-pragmas"])
        if res2.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + res.stderr + "\n" + res2.stderr)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

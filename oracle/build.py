"""Build the CPU oracle (plain C, gcc) into oracle/liboracle*.so.

Test infrastructure: only tests/, the smoke check and the bench's CPU legs use
the result.  The flags keep every float operation a single IEEE binary32 /
binary64 operation: no contraction into FMA, no fast-math.

liboracle_omp.so is the same source built with -fopenmp: the GEMM's rows are
shared out between threads (each output element is still computed by one
thread in the source's order, so its values equal the single-threaded
library's).  The full-size parity tests use it; the bench's CPU baseline
times the single-threaded library.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fexcess-precision=standard", "-Wall", "-Wextra"]


def lib_path(mutant: int = 0, omp: bool = False) -> str:
    if omp:
        assert mutant == 0, "the threaded build is of the real oracle only"
        return os.path.join(HERE, "liboracle_omp.so")
    name = "liboracle.so" if mutant == 0 else f"liboracle_mut{mutant}.so"
    return os.path.join(HERE, name)


def build(mutant: int = 0, force: bool = False, omp: bool = False) -> str:
    out = lib_path(mutant, omp)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SRC)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, *(["-fopenmp"] if omp else []), f"-DORC_MUTANT={mutant}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
    print(build(force=True, omp=True))

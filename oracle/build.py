"""Compile the C oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc, -O2, no fast-math, no fp contraction (products are exact either
way, but the sums must be plain fp32 adds), OpenMP when the compiler has it.
Runs on x86_64 and aarch64 alike: no architecture flags.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_SRC = os.path.join(HERE, "w8_oracle.c")
ORACLE_SO = os.path.join(HERE, "liboracle.so")


def build_oracle(verbose: bool = False, src: str = ORACLE_SRC, out: str = ORACLE_SO) -> str:
    tmp = out + ".tmp"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", src, "-o", tmp, "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:4] + extra + base[4:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, out)
            if verbose:
                print(" ".join(cmd))
            return out
    raise RuntimeError("could not compile the oracle:\n" + r.stderr)


if __name__ == "__main__":
    print(build_oracle(verbose=True))

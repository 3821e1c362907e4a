"""Builds the CPU oracle (plain C, gcc) into ``oracle/liboracle.so``.

Test infrastructure: the library under test never links or loads this.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "conv_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the oracle if the shared library is missing or stale; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-O2", "-std=c11", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp"]
    # OpenMP over (n, k) when the compiler has it; the loops are the same either way.
    for extra in (["-fopenmp"], []):
        cmd = base[:2] + extra + base[2:]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode == 0:
            os.replace(LIB + ".tmp", LIB)
            if verbose:
                print(" ".join(cmd))
            return LIB
    raise RuntimeError("oracle build failed:\n" + res.stderr)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

"""Compile the CPU oracle (oracle/oracle.c) into oracle/liboracle.so.

Test infrastructure: the oracle is a checker, not part of the library.
Plain gcc, -O2, no floating-point contraction and no fast-math, so every
double addition is a separately rounded IEEE operation.  OpenMP is used
when the compiler accepts -fopenmp; otherwise the build is single-threaded.
"""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def _compile(flags):
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found to build the oracle")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", *flags, SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        if os.path.exists(tmp):
            os.unlink(tmp)
        return False, r.stderr
    os.replace(tmp, LIB)
    return True, ""


def build(force=False):
    """Build liboracle.so if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    ok, err = _compile(["-fopenmp"])
    if not ok:
        ok, err = _compile([])
    if not ok:
        raise RuntimeError("oracle build failed:\n" + err)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

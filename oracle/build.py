"""Compile the C oracle into ``oracle/liboracle.so``.

Test infrastructure: the oracle is compiled here so that tests and the CPU
baseline can load it, never so that the product path can.  Plain gcc, no
-ffast-math and no FMA contraction, so that ``x / T`` stays a correctly rounded
binary32 division.  OpenMP is used when the compiler has it (rows in parallel);
without it the same code runs single-threaded.
"""
import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def _compile(flags, out):
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", *flags, SRC, "-o", out, "-lm"]
    return subprocess.run(cmd, capture_output=True, text=True)


def build(force=False, verbose=False):
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(os.path.join(HERE, "oracle.h"))):
        return LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
    os.close(fd)
    try:
        res = _compile(["-fopenmp"], tmp)
        if res.returncode != 0:
            res = _compile([], tmp)
        if res.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + res.stderr)
        if verbose and res.stderr:
            print(res.stderr)
        os.replace(tmp, LIB)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

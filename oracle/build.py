"""Build the float64 CPU oracle (test infrastructure only).

Compiles ``oracle.c`` with the host C compiler into ``liboracle.so`` beside
it.  Plain C with OpenMP; no CUDA, no BLAS, nothing shared with the CUDA
library.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(src=SRC, out=LIB, extra_flags=(), quiet=True):
    """Compile ``src`` into the shared library ``out``; return ``out``."""
    if (src == SRC and out == LIB and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    cc = os.environ.get("CC", "gcc")
    tmp = out + ".tmp%d" % os.getpid()
    cmd = [cc, "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", *extra_flags, src, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + " ".join(cmd) + "\n" + res.stderr)
    os.replace(tmp, out)
    if not quiet:
        print("built", out)
    return out


if __name__ == "__main__":
    build(quiet=False)
    sys.exit(0)

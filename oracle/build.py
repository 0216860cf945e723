"""Compile the fp64 attention oracle (test infrastructure) into a shared library.

Run as a script (``python oracle/build.py``) or call ``build()``.  The library
lands beside its source as ``liboracle_attn.so``.  OpenMP is used when the
compiler supports it; otherwise the oracle is built single-threaded.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
LIB = os.path.join(HERE, "liboracle_attn.so")


def build(src=SRC, lib=LIB, force=False, quiet=True):
    """Build ``lib`` from ``src`` unless it is already newer than the source."""
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(src):
        return lib
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", src, "-o", lib + ".tmp"]
    for extra in (["-fopenmp"], []):
        cmd = base[:4] + extra + base[4:] + ["-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(lib + ".tmp", lib)
            return lib
        if not quiet:
            sys.stderr.write(r.stderr)
    raise RuntimeError("oracle build failed: " + r.stderr)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, quiet=False))

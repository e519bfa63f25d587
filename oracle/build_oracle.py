"""Build step for the FP64 CPU oracle (test infrastructure only).

Compiles ``qsa_oracle.c`` with the host C compiler into ``libqsa_oracle.so``
next to it.  Plain ``-O2`` without fast-math, so sums keep their written order.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qsa_oracle.c")
LIB = os.path.join(HERE, "libqsa_oracle.so")


def build(force: bool = False, src: str = SRC, out: str = LIB, defines=()) -> str:
    """Compile the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)
            and os.path.getmtime(out) >= os.path.getmtime(os.path.join(HERE, "qsa_oracle.h"))):
        return out
    cc = os.environ.get("CC", "gcc")
    cmd = [cc, "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-I", HERE,
           *[f"-D{d}" for d in defines], "-o", out + ".tmp", src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

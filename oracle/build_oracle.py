"""Build the CPU oracle (plain C, gcc) into a shared library.

Test infrastructure only: tests/, __graft_entry__ and bench.py's CPU
baseline are the only users.  -ffp-contract=off keeps gcc from fusing any
multiply-add the source does not write as fmaf (gcc fuses by default on
aarch64), so the oracle gives the same bits on x86-64 and Arm hosts.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "afd_oracle.c")
LIB = os.path.join(HERE, "liborc_afd.so")


def build(out=LIB, plant=0, quiet=True):
    """Compile afd_oracle.c; plant > 0 builds a deliberately wrong variant."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", f"-DORC_PLANT={int(plant)}",
           "-o", out, SRC, "-lm"]
    subprocess.run(cmd, check=True,
                   stdout=subprocess.DEVNULL if quiet else None)
    return out


def ensure_built():
    if (not os.path.exists(LIB)
            or os.path.getmtime(LIB) < os.path.getmtime(SRC)):
        build()
    return LIB


if __name__ == "__main__":
    print(build(quiet=False))

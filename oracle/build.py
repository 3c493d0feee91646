"""Build the plain-C CPU oracle into ``oracle/liboracle.so`` (single-threaded)
and ``oracle/liboracle_omp.so`` (the same source with -fopenmp: independent
rows and tokens spread over threads, every sum in the same order).

Test infrastructure only: the library never links or loads the oracle.
Flags keep IEEE semantics: no fast-math, no FMA contraction.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "coli_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")
LIB_OMP = os.path.join(HERE, "liboracle_omp.so")
FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
         "-Wno-unknown-pragmas"]


def _build(out, extra, force):
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SRC)):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    cc = os.environ.get("CC", "gcc")
    subprocess.check_call([cc, *FLAGS, *extra, SRC, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build_oracle(force: bool = False) -> str:
    """Compile the single-threaded oracle if missing or older than its source."""
    return _build(LIB, [], force)


def build_oracle_omp(force: bool = False) -> str:
    """Compile the OpenMP build of the same source."""
    return _build(LIB_OMP, ["-fopenmp"], force)


if __name__ == "__main__":
    print(build_oracle(force=True))
    print(build_oracle_omp(force=True))

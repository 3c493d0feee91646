"""Build the plain-C CPU oracle into ``oracle/liboracle.so``.

Test infrastructure only: the library never links or loads the oracle.
Flags keep IEEE semantics: no fast-math, no FMA contraction.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "coli_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")
FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build_oracle(force: bool = False) -> str:
    """Compile the oracle if the shared object is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cc = os.environ.get("CC", "gcc")
    subprocess.check_call([cc, *FLAGS, SRC, "-o", tmp, "-lm"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))

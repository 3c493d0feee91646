"""The diagnostic bounds-checked build (-DCOLI_CHECK, libcoli_check.so): every
index a kernel derives from data (expert ids, union and route lists, token ids
of the batched grouping) is checked against its buffer and reported through
COLI_FLAG_BOUNDS.  The library is built here and the cases of
checked_build_cases.py run against it in a child process (COLI_LIBRARY=check):
parity with the oracle and no flag on any path."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_runs_clean():
    from int4_expert_ffn_gb300 import build as b
    lib = b.build(variant="check")
    assert lib.endswith("libcoli_check.so") and os.path.exists(lib)
    env = dict(os.environ, COLI_LIBRARY="check")
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_build_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "all cases passed" in r.stdout

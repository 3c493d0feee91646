import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def parse_golden(path):
    """Parse a golden quantiser fixture: list of dicts with cols, w, bytes, scales."""
    cases, cur = [], None
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0], "w": [], "bytes": [], "scales": []}
            elif key == "cols":
                cur["cols"] = int(vals[0])
            elif key == "w":
                cur["w"].append([float(v) for v in vals])
            elif key == "bytes":
                cur["bytes"].append([int(v, 16) for v in vals])
            elif key == "scales":
                cur["scales"].append([int(v, 16) for v in vals])
            elif key == "end":
                cases.append(cur)
                cur = None
            else:
                raise ValueError("bad golden line: %r" % line)
    return cases

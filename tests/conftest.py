import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Parse a `key = values` golden file into {key: [list of float rows]}."""
    import math

    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = (s.strip() for s in line.split("=", 1))
            row = []
            for tok in vals.split():
                row.append(math.log(float(tok[2:])) if tok.startswith("ln") else float(tok))
            out.setdefault(key, []).append(row)
    return out


@pytest.fixture(scope="session")
def golden():
    return read_golden

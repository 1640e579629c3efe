import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (seconds to minutes)")


GOLDEN = os.path.join(HERE, "golden")


def read_golden(name):
    """Parse a golden text fixture: '#' lines are comments; other lines are 'tag values...'."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, *vals = line.split()
            rows.append((tag, [int(v, 0) for v in vals]))
    return rows


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.lib()
    return oracle

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def load_golden(name):
    """Parse a tests/golden fixture: '# ...' comments, 'key: v v v' lines, and
    'key:' followed by bare lines (kept as strings)."""
    out = {}
    key = None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                key = k.strip()
                v = v.strip()
                if v:
                    vals = v.split()
                    try:
                        out[key] = [int(x) for x in vals]
                    except ValueError:
                        out[key] = [float(x) for x in vals]
                    key = None
                else:
                    out[key] = []
            elif key is not None:
                out[key].append(line)
    return out


@pytest.fixture
def golden():
    return load_golden

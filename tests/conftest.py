import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: large-size case (minutes of CPU time in the oracle)")


def read_golden(name):
    """Parse a tests/golden fixture: '# ...' comments, then 'key v v v ; v v ...' lines.

    Values are returned as lists of rows (';' separates rows); each value stays a string so the
    caller decides how to read it (decimal, hex code, 'inf')."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            out[key] = [row.split() for row in rest.split(";")]
    return out

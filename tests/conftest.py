import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a) and the built libtq.so")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(v):
    try:
        return int(v, 0)
    except ValueError:
        return float(v)


def read_golden(name):
    """Read a fixture: '#' lines are comments (citations); other lines are 'key: values'."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            out[key.strip()] = [_num(v) for v in val.split()]
    return out

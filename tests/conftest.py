import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


def golden_path(name: str) -> str:
    return os.path.join(TESTS, "golden", name)


def read_golden(name: str):
    """Parse a golden fixture: '#' comments, 'key value...' lines and bare numeric rows."""
    kv, rows = {}, []
    with open(golden_path(name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            try:
                rows.append([float(p) for p in parts])
            except ValueError:
                kv.setdefault(parts[0], []).append(parts[1:])
    return kv, rows

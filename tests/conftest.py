"""Shared test set-up.

Tests marked ``gpu`` need a CUDA device and the built CUDA library; all other
tests run on the CPU (the oracle, the input generator, host-side logic and
the C-ABI export check)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: large sizes, still bounded to a few seconds of oracle work")


def read_golden(name):
    """Parse a golden fixture: '#' comment lines, then '<key> <values...>'."""
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append([float(v) for v in vals])
    return rows

"""Shared pytest configuration.

Markers: ``gpu`` marks tests that need a CUDA device (parity tests through the
C ABI); everything else runs on a CPU-only machine.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


def read_golden(name):
    """Rows of a ``tests/golden`` fixture: '|'-separated records or 'key = value' lines."""
    path = os.path.join(ROOT, "tests", "golden", name)
    rows, kv = [], {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if "|" in line:
                rows.append([c.strip() for c in line.split("|")])
            elif "=" in line:
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
    return rows, kv

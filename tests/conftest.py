"""Shared pytest set-up: the ``gpu`` marker and the repository root on sys.path."""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name: str) -> dict[str, list[float]]:
    """Parse a ``key: v v v`` fixture; '#' starts a comment line."""
    out: dict[str, list[float]] = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, vals = line.split(":", 1)
            out[key.strip()] = [float(v) for v in vals.split()]
    return out


@pytest.fixture(scope="session")
def worked_example():
    return read_golden("worked_example_p4.txt")

"""Shared test set-up: the ``gpu`` marker, import paths and golden-file parsing."""
from __future__ import annotations

import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
GOLDEN = Path(__file__).resolve().parent / "golden"
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300); parity tests proper")


def read_golden(name: str) -> dict:
    """Parse a golden file: '#' lines are comments, data lines are 'key: value'."""
    out = {}
    for line in (GOLDEN / name).read_text(encoding="utf-8").splitlines():
        s = line.strip()
        if not s or s.startswith("#"):
            continue
        key, _, val = s.partition(":")
        out[key.strip()] = val.strip()
    return out


def ints(s: str) -> list:
    return [int(t, 0) for t in s.split()]


@pytest.fixture(scope="session")
def golden():
    return read_golden

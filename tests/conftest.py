"""Shared pytest set-up: the ``gpu`` marker, the repository root on sys.path,
and session-scoped builds of the oracle and of the CUDA library."""
from __future__ import annotations

import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU; parity tests through the C ABI")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load_library()

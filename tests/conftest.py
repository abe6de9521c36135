import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

GOLDEN = Path(__file__).resolve().parent / "golden"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload; minutes of host time")


@pytest.fixture(scope="session")
def oracle():
    import oracle as o

    o.load()
    return o


@pytest.fixture(scope="session")
def golden():
    import json

    def _load(name):
        with open(GOLDEN / name) as f:
            return json.load(f)

    return _load

import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

GOLDEN = Path(__file__).resolve().parent / "golden"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs an sm_103 GPU and the built libgtp.so")


@pytest.fixture(scope="session")
def golden():
    import json

    def load(name):
        return json.loads((GOLDEN / name).read_text())
    return load

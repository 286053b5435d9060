import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def read_golden(name):
    """Parse a tests/golden facts file: ``key = value | citation`` lines."""
    facts = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0] if line.lstrip().startswith("#") else line
            if "=" not in line:
                continue
            key, rest = line.split("=", 1)
            value = rest.split("|", 1)[0].strip()
            facts[key.strip()] = value
    return facts


@pytest.fixture(scope="session")
def golden_facts():
    return read_golden("pages_facts.txt")

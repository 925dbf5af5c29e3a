import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (run on the GB300 box)")
    config.addinivalue_line("markers", "slow: long CPU test")


def page_facts():
    """Parse tests/golden/page_facts.txt into a dict of strings."""
    facts = {}
    with open(os.path.join(ROOT, "tests", "golden", "page_facts.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if "=" in line:
                k, v = line.split("=", 1)
                facts[k.strip()] = v.strip()
    return facts


@pytest.fixture(scope="session")
def facts():
    return page_facts()

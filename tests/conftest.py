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


def pytest_terminal_summary(terminalreporter):
    """Print how close each parity case came to its bound (worst error / bound)."""
    mod = sys.modules.get("parity")
    report = getattr(mod, "REPORT", None) if mod else None
    if not report:
        return
    tr = terminalreporter
    tr.section("parity: worst |C_gpu - C_exact| / bound per case")
    for name, worst, count in sorted(report, key=lambda x: -x[1]):
        tr.write_line(f"{worst:10.3e}  {count:>12d} elements  {name}")
    path = os.environ.get("PARITY_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            for name, worst, count in report:
                f.write(json.dumps({"test": name, "worst_ratio": worst, "elements": count}) + "\n")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running oracle checks")


def read_golden(name):
    """Parse a tests/golden fixture: '# ...' lines are its citation, the rest
    'key: values' pairs (values split on whitespace) or raw rows."""
    path = os.path.join(ROOT, "tests", "golden", name)
    fields, rows = {}, []
    with open(path, encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, sep, val = line.partition(":")
            if sep and key.strip().isidentifier():
                fields[key.strip()] = val.split()
            else:
                rows.append(line.split())
    return fields, rows

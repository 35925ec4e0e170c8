"""Test configuration: the ``gpu`` marker and shared helpers.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything
else runs on a CPU-only machine.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libpkv.so")


def load_golden(name):
    """Parse a fixture: '# ...' comments; 'key v v ; v v' rows; 'case NAME' starts a new case.

    Returns {case: {key: list-of-rows}} where each row is a list of floats; keys
    before any 'case' line land in case ''.
    """
    cases = {"": {}}
    cur = cases[""]
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = cases.setdefault(rest.strip(), {})
                continue
            rows = [[float(x) for x in part.split()] for part in rest.split(";")]
            cur[key] = rows
    return cases


@pytest.fixture
def golden():
    return load_golden

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


class ExceptionLog:
    """Session-wide log of integer disagreements excused by the 1e-5 rule.

    A GPU/oracle disagreement on an integer output is excused only when the
    oracle's |u - alpha| at the first differing decision, or its inverse-CDF
    margin at the differing draw, is <= 1e-5.  The excused count must stay
    <= 1e-5 of all verified rows checked in the session.
    """

    def __init__(self):
        self.rows = 0
        self.entries = []

    def add_rows(self, n):
        self.rows += int(n)

    def excuse(self, where, margin):
        self.entries.append((where, float(margin)))
        print(f"[parity exception] {where}: margin {margin:.3e}")


_LOG = ExceptionLog()


@pytest.fixture(scope="session")
def exception_log():
    return _LOG


def pytest_sessionfinish(session, exitstatus):
    if _LOG.rows:
        n = len(_LOG.entries)
        print(f"\n[parity] rows checked {_LOG.rows}, excused disagreements {n}")
        for where, margin in _LOG.entries:
            print(f"[parity] excused: {where}: margin {margin:.3e}")
        if n > 1e-5 * _LOG.rows:
            print("[parity] FAIL: excused disagreements exceed 1e-5 of rows")
            session.exitstatus = 1

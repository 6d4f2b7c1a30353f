import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_terminal_summary(terminalreporter):
    """Largest per-(query, head) attention error of every GPU parity check, by label."""
    from attn_check import RECORDS
    if not RECORDS:
        return
    worst = {}
    for label, per, whole in RECORDS:
        key = label.split("#")[0]
        w = worst.get(key, (0.0, 0.0, 0))
        worst[key] = (max(w[0], per), max(w[1], whole), w[2] + 1)
    terminalreporter.write_sep("-", "attention error per (query, head) vector, worst per label")
    for key in sorted(worst):
        per, whole, n = worst[key]
        terminalreporter.write_line(f"{key:60s} per-head max {per:.3e}  whole max {whole:.3e}  ({n} checks)")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


def pytest_terminal_summary(terminalreporter):
    """Counts of near-tie routing differences of the end-to-end layer tests: a
    token may route differently from the oracle only where the oracle's keys
    nearly tie (relative gap < 1e-4); every such token is counted here."""
    helpers = sys.modules.get("gpu_helpers")
    log = getattr(helpers, "NEAR_TIE_LOG", None)
    if not log:
        return
    terminalreporter.section("near-tie routing (tokens / oracle near-ties / routed differently / compared)")
    for name, tokens, near, diff, compared in log:
        terminalreporter.write_line(f"{name}: {tokens} / {near} / {diff} / {compared}")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def pytest_terminal_summary(terminalreporter):
    """Print the full-size element-wise parity lines, if any test recorded one."""
    util = sys.modules.get("gpu_util")
    lines = getattr(util, "PARITY_LOG", None) if util else None
    if lines:
        terminalreporter.section("element-wise parity against the oracle")
        for line in lines:
            terminalreporter.write_line(line)


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle

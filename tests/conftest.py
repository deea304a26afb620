import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")

import oracle_check  # noqa: E402  (tests/ is on sys.path for its own modules)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


@pytest.fixture(autouse=True)
def _bar_record(request):
    """Name the running test for the per-column bar record."""
    oracle_check._current[0] = request.node.nodeid
    yield
    oracle_check._current[0] = None


def pytest_terminal_summary(terminalreporter):
    if not oracle_check.WORST:
        return
    worst = sorted(oracle_check.WORST.items(), key=lambda kv: -kv[1])
    terminalreporter.write_line(f"fraction of the 4e-3 per-column bar used: max {worst[0][1]:.3f} "
                                f"over {len(worst)} tests; largest:")
    for name, used in worst[:12]:
        terminalreporter.write_line(f"  {used:.3f}  {name}")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload, minutes of CPU oracle time")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """The top-K near-tie swaps the parity tests saw (each one bounded by
    check_topk's rule), per test with any, and in total."""
    parity = sys.modules.get("parity")
    log = getattr(parity, "TIE_LOG", None) if parity else None
    if not log:
        return
    swaps = sum(v[0] for v in log.values())
    rows = sum(v[1] for v in log.values())
    terminalreporter.write_line(f"top-K near-tie swaps: {swaps} over {rows} token rows "
                                f"checked against whole oracle rows")
    for name, (sw, rw) in sorted(log.items()):
        if sw:
            terminalreporter.write_line(f"  {name}: {sw} swaps over {rw} rows")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Per comparison of the GPU parity tests: elements compared, the largest
    absolute error and the largest |err| / (2e-3 + 1e-2 |ref|) (the bar is 1)."""
    mod = sys.modules.get("gpu_harness")
    log = getattr(mod, "PARITY_LOG", None) if mod else None
    if not log:
        return
    tr = terminalreporter
    tr.section("parity against the fp64 oracle")
    tr.write_line(f"{'test / output':<92} {'elements':>11} {'max|err|':>10} {'err/bar':>8}")
    for test, what, n, e, r in log:
        name = f"{test.split('::', 1)[-1]} / {what}"
        tr.write_line(f"{name[:92]:<92} {n:>11} {e:>10.3e} {r:>8.3f}")

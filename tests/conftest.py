import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


def pytest_terminal_summary(terminalreporter):
    """Attention parity diagnostics: the largest errors, also in bf16 ulps."""
    mod = sys.modules.get("tests._gpu")
    log = getattr(mod, "ULP_LOG", None) if mod else None
    if not log:
        return
    terminalreporter.write_line(
        f"attention parity: {len(log)} comparisons, max |d| {max(r[1] for r in log):.2e}, "
        f"max mean |d| {max(r[2] for r in log):.2e}; the largest errors, with each in bf16 "
        f"ulps of the rounded oracle value where it occurs:")
    for what, mx, mean, ulps, _, _ in sorted(log, key=lambda r: -r[1])[:5]:
        terminalreporter.write_line(f"  max|d| {mx:.2e} ({ulps:.1f} ulps)  mean|d| {mean:.2e}  {what}")
    terminalreporter.write_line(
        "the largest mean errors, each also against the oracle rounded to bf16 (RNE, as the "
        "kernels round their outputs), which takes out the output rounding:")
    for what, mx, mean, _, rmx, rmean in sorted(log, key=lambda r: -r[2])[:3]:
        terminalreporter.write_line(
            f"  mean|d| {mean:.2e} max|d| {mx:.2e}; vs rounded oracle: mean {rmean:.2e} "
            f"max {rmx:.2e}  {what}")

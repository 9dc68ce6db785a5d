import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libfattn")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the parity statistics the full-size tests asked to report (how
    many elements needed the output-rounding allowance, largest errors)."""
    try:
        from tests.parity import REPORTED
    except Exception:
        return
    if not REPORTED:
        return
    terminalreporter.section("parity against the fp64 oracle (full-size workloads)")
    for what, st in REPORTED:
        line = "%s: %d elements, max |dO| %.3e, mean |dO| %.3e, over the gate %d" % (
            what, st["n"], st["max_abs"], st["mean_abs"], st["n_over_gate"])
        if st["n_over_gate"]:
            line += " (max |dO| among them %.3e, max %.0f ulp from the rounded oracle)" % (
                st["over_gate_max_abs"], st["over_gate_max_ulps_from_rounded_oracle"])
        if "lse_max_abs" in st:
            line += ", max |dLSE| %.3e" % st["lse_max_abs"]
        terminalreporter.write_line(line)

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libpsk.so")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter):
    """Selected-id parity: how many (sequence, head) rows were compared with the oracle and how
    many differed at the cutoff within the 1e-6-relative near-tie band (each one listed). With
    PSK_NEAR_TIES_JSON set, the same record is written to that file."""
    parity = sys.modules.get("parity")
    if parity is None or not parity.SELECTION_LOG["units"]:
        return
    log = parity.SELECTION_LOG
    terminalreporter.write_line(f"selected-id parity: {log['units']} rows compared with the oracle, "
                                f"{len(log['near_ties'])} near ties at the cutoff (within 1e-6 relative, accepted)")
    for t in log["near_ties"]:
        terminalreporter.write_line(f"  near tie: {t['test']} pages {t['pages']} rel. to cutoff {t['rel_to_cutoff']}")
    path = os.environ.get("PSK_NEAR_TIES_JSON")
    if path:
        import json
        with open(path, "w") as f:
            json.dump(log, f, indent=1)

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU-side oracle work")


@pytest.fixture(scope="session")
def cuda_ok():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Slot-set parity counts of every workload the GPU tests checked against the
    oracle: sampled tokens, mismatches a near-tie does not excuse (the tests fail on
    any), and mismatches excused because the oracle's gap between the W-th and
    (W+1)-th combined score is below 1e-5. One JSON line per workload and query kind."""
    mod = sys.modules.get("tests.sdm_testlib")
    recs = getattr(mod, "ADDRESS_REPORT", None) if mod is not None else None
    if not recs:
        return
    terminalreporter.section("slot-set parity (near-ties counted)")
    for r in recs:
        terminalreporter.write_line(json.dumps(r))

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(scope="session")
def orc():
    from oracle import oracle
    return oracle.default()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Counts of the sampling comparisons: requests compared with the oracle, requests
    excluded on the 1e-6 decision margin (with the bound asserted), and bonus draws within
    1e-6 of a CDF boundary (checked against the oracle's draw window). Also written as JSON
    to the path in SPEC_PARITY_LOG, when set."""
    parity = sys.modules.get("parity")
    recs = getattr(parity, "RECORDS", None)
    if not recs:
        return
    tr = terminalreporter
    tr.section("sampling parity against the oracle")
    tot = dict(requests=0, excluded=0, near=0)
    for r in recs:
        tr.write_line(f"{r['test']}: {r['requests']} requests, {r['excluded']} excluded on the "
                      f"decision margin (bound {r['bound']}), {r['near']} near a CDF boundary")
        for k in tot:
            tot[k] += r[k]
    tr.write_line(f"total: {len(recs)} comparisons, {tot['requests']} requests, "
                  f"{tot['excluded']} excluded, {tot['near']} near a CDF boundary")
    path = os.environ.get("SPEC_PARITY_LOG")
    if path:
        import json
        with open(path, "w") as f:
            json.dump({"comparisons": recs, "total": tot}, f, indent=1)

import os
import sys

import pytest

TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)
for _p in (ROOT, TESTS):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU or GPU case")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Table of the parity errors the GPU tests measured (see _margins.py)."""
    import json

    import _margins
    recs = _margins.RECORDS
    if not recs:
        return
    tr = terminalreporter
    tr.section("parity margins: max|gpu - oracle| / max|oracle|")
    worst = {}
    for r in recs:
        key = (r["test"] + ": " + r["case"], r["quantity"])
        if key not in worst or r["err"] > worst[key]["err"]:
            worst[key] = r
    for (case, qty), r in sorted(worst.items()):
        head = r["tol"] / r["err"] if r["err"] > 0 else float("inf")
        tr.write_line(f"{r['err']:10.3e}  tol {r['tol']:.0e}  x{head:9.1f}  {qty:6s} {case}")
    path = os.environ.get("KDA_PARITY_JSON")
    if path:
        with open(path, "w") as f:
            json.dump(list(worst.values()), f, indent=1)

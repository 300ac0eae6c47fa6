"""Measured parity margins of the GPU tests.

Every GPU parity check records the error it measured, max|x_gpu - x_ref| /
max|x_ref| against the float64 oracle, next to the tolerance it asserts.
The session prints them as a table at the end of the run and, when the
environment variable KDA_PARITY_JSON names a file, writes them there as
JSON, so that the achieved errors and their headroom are on record, not
only the pass/fail outcome.
"""
import os

RECORDS = []


def record(case, quantity, err, tol):
    """Note one measured error (a float) of `quantity` ("o", "hT", ...) in
    `case`, with the id of the test that measured it."""
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0].split("::")[-1]
    RECORDS.append({"case": str(case), "quantity": str(quantity), "err": float(err),
                    "tol": float(tol), "test": test})
    return err


def case_name(w, path=None):
    """Short description of a prefill workload (and path) for the table."""
    s = (f"{w.name} B={w.B} H={w.H} T={w.T} dk={w.dk} dv={w.dv} C={w.C} {w.dtype} "
         f"{w.alpha}")
    return s if path is None else f"{s} [{path}]"

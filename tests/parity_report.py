"""Achieved parity errors of the GPU tests, collected while they run.

A test calls record(case, **metrics) with the errors it measured against the oracle;
when the environment variable FDMA_PARITY_REPORT names a file, the session writes
every recorded case there as JSON at the end (tests/conftest.py).  Nothing is written
otherwise."""
import json
import os

REPORT = {}


def record(case: str, **metrics):
    entry = REPORT.setdefault(case, {})
    for k, v in metrics.items():
        entry[k] = float(v) if v is not None else None


def write():
    path = os.environ.get("FDMA_PARITY_REPORT")
    if path and REPORT:
        with open(path, "w") as f:
            json.dump(REPORT, f, indent=1, sort_keys=True)

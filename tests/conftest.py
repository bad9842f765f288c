import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built libtq.so")
    config.addinivalue_line("markers", "slow: full-size workload, minutes on the GPU box")


def pytest_terminal_summary(terminalreporter):
    """Report the code / norm comparison counts of the GPU parity tests
    (coordinates within 1e-5 of a decision boundary, mismatches) and the
    other reported quantities, one line per comparison."""
    try:
        from parity_util import RECORDS
    except Exception:
        return
    if not RECORDS:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity counts (%d comparisons)" % len(RECORDS))
    tot = {}
    for r in RECORDS:
        keys = [k for k in r if k != "label"]
        tr.write_line("%-28s %s" % (r["label"][:28], " ".join("%s=%s" % (k, r[k]) for k in keys)))
        for k in keys:
            if isinstance(r[k], int) and k != "bits":
                tot[k] = tot.get(k, 0) + r[k]
    if tot.get("coords"):
        tr.write_line("total: %s; code mismatch fraction %.2e, norm mismatch fraction %.2e" % (
            " ".join("%s=%d" % kv for kv in sorted(tot.items())), tot.get("code_mismatch", 0) / tot["coords"],
            tot.get("norm_mismatch", 0) / max(1, tot.get("vectors", 0))))

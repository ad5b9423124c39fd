import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running parity case")


def pytest_terminal_summary(terminalreporter):
    """The GPU parity errors next to the bf16 rounding floor of each case."""
    try:
        from tests import helpers
    except Exception:   # pragma: no cover - helpers not imported in this run
        return
    if not helpers.RESULTS:
        return
    tr = terminalreporter
    tr.section("parity against the fp64 oracle (GPU error | bf16 floor of the oracle)")
    tr.write_line(f"{'case':60s} {'rel_frob':>10s} {'max_abs':>10s} | {'rel_frob':>10s} {'max_abs':>10s}")
    for what, rf, ma, frf, fma in helpers.RESULTS:
        tr.write_line(f"{what[:60]:60s} {rf:10.3e} {ma:10.3e} | {frf:10.3e} {fma:10.3e}")
    # G3_PARITY_JSON=<path>: the same table as one JSON record per case.
    path = os.environ.get("G3_PARITY_JSON")
    if path:
        recs = [{"case": what, "rel_frob": rf, "max_abs": ma, "floor_rel_frob": frf,
                 "floor_max_abs": fma, "tol_rel_frob": helpers.REL_FROB,
                 "tol_max_abs": helpers.MAX_ABS} for what, rf, ma, frf, fma in helpers.RESULTS]
        with open(path, "w") as f:
            json.dump(recs, f, indent=1)
        tr.write_line(f"parity records: {path}")

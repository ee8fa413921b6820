import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the kernels)")
    config.addinivalue_line("markers", "slow: full-size workload")


def pytest_collection_modifyitems(config, items):
    # gpu tests must find a GPU; on a machine without one they are skipped
    # only when they were not explicitly selected with -m gpu
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    markexpr = config.getoption("-m") or ""
    if "gpu" in markexpr and "not gpu" not in markexpr:
        return  # fail loudly: gpu tests were asked for on a box without one
    skip = pytest.mark.skip(reason="no CUDA GPU on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    # one line per FP8 code comparison that used rounding-boundary
    # exemptions, plus the totals (tests/parity.py records them); also
    # written as JSON when RN_EXEMPTIONS_JSON names a file
    try:
        import parity
    except Exception:  # pragma: no cover
        return
    recs = getattr(parity, "EXEMPTIONS", [])
    if not recs:
        return
    tr = terminalreporter
    tr.section("FP8 rounding-boundary exemptions")
    tot = {"elements": 0, "mismatches": 0, "literal": 0, "widened_only": 0}
    for r in recs:
        for k in tot:
            tot[k] += r[k]
        if r["mismatches"]:
            tr.write_line(f"{r['what']:>28s}: {r['mismatches']:8d} of {r['elements']:11d} "
                          f"({r['mismatches'] / r['elements']:.2e}); within 1e-6|p| {r['literal']}, "
                          f"widened only {r['widened_only']}")
    tr.write_line(f"{'all ' + str(len(recs)) + ' comparisons':>28s}: {tot['mismatches']:8d} of "
                  f"{tot['elements']:11d} ({tot['mismatches'] / max(1, tot['elements']):.2e}); "
                  f"within 1e-6|p| {tot['literal']}, widened only {tot['widened_only']}")
    path = os.environ.get("RN_EXEMPTIONS_JSON")
    if path:
        import json
        with open(path, "w") as f:
            json.dump({"records": recs, "total": tot}, f)

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """GEMM parity statistics of the run: per test the largest fp32 rel-L2,
    the largest bf16 ulp distance, and how many elements passed only by the
    fp32 accumulation bound (y ~ 0 after cancellation) rather than 1 ulp."""
    try:
        from parity_util import STATS
    except Exception:  # pragma: no cover
        return
    if not STATS:
        return
    tr = terminalreporter
    per = {}
    for s in STATS:
        d = per.setdefault(s["test"], {"calls": 0, "elements": 0, "floor_used": 0, "max_ulp": 0, "rel_l2": 0.0})
        d["calls"] += 1
        d["elements"] += s["elements"]
        d["floor_used"] += s["floor_used"]
        d["max_ulp"] = max(d["max_ulp"], s["max_ulp"])
        d["rel_l2"] = max(d["rel_l2"], s["rel_l2"])
    tr.write_sep("-", "GEMM parity vs oracle (per test: compares, elements, max rel-L2, max bf16 ulp, floor used)")
    for name, d in per.items():
        tr.write_line(f"{name}: {d['calls']} x, {d['elements']} el, rel-L2 {d['rel_l2']:.2e}, "
                      f"ulp {d['max_ulp']}, floor {d['floor_used']}")
    el = sum(d["elements"] for d in per.values())
    fl = sum(d["floor_used"] for d in per.values())
    tr.write_line(f"GEMM parity total: {len(STATS)} compares, {el} elements, max rel-L2 "
                  f"{max(d['rel_l2'] for d in per.values()):.2e}, max ulp {max(d['max_ulp'] for d in per.values())}, "
                  f"floor used on {fl} elements ({fl / max(el, 1):.2e})")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running case")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Rows the GPU parity tests excluded at a boundary, per case (the
    comparisons bound them; this prints the counts)."""
    H = sys.modules.get("gpu_helpers")
    if H is None or not getattr(H, "BOUNDARY_LOG", None):
        return
    agg = {}
    for name, st in H.BOUNDARY_LOG:
        a = agg.setdefault(name, dict(calls=0, rows=0, topp_boundary=0, cdf_boundary=0))
        a["calls"] += 1
        for k in ("rows", "topp_boundary", "cdf_boundary"):
            a[k] += st.get(k, 0)
    terminalreporter.write_sep("-", "rows excluded at a boundary (top-p mass within 1e-5 of p; "
                                    "u within 1e-6 of a CDF boundary)")
    for name, a in sorted(agg.items()):
        terminalreporter.write_line(f"{name}: {a['calls']} comparisons, {a['rows']} rows, "
                                    f"top-p boundary {a['topp_boundary']}, "
                                    f"CDF boundary {a['cdf_boundary']}")

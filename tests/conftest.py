import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def _gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _gpu_available():
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the parity margins the full-size GPU tests recorded."""
    try:
        from tests import kda_testlib as tl
    except Exception:
        return
    tr = terminalreporter
    if tl.GRAD_MARGINS:
        tr.section("KDA backward margins (rel-RMS of each gradient against the fp64 autograd oracle)")
        tr.write_line("bound: rel-RMS <= 1e-3 and max-abs <= 1e-2 max|ref| per gradient")
        for tag, errs in tl.GRAD_MARGINS:
            tr.write_line(f"{tag:<22} " + "  ".join(f"d{k} {v:.1e}" for k, v in errs.items()))
    if not tl.MARGINS:
        return
    tr.section("KDA parity margins (full-size workloads, every unit, against the fp64 oracle)")
    tr.write_line(f"bounds: out rel-RMS <= {tl.OUT_RMS:g}, out max-abs <= {tl.OUT_MAXABS:g} max|ref|, "
                  f"final-state rel-RMS <= {tl.STATE_RMS:g}")
    for tag, r, m, w, st in tl.MARGINS:
        sts = "-" if st is None else f"{st:.3e}"
        tr.write_line(f"{tag:<28} out rel-RMS {r:.3e}  max-abs/max|ref| {m:.3e}  "
                      f"worst unit rel-RMS {w:.3e}  state rel-RMS {sts}")

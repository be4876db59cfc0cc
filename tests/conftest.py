import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity margins of the labelled comparisons (full-size workloads, strong decay): per label,
    each output's raw max|x - ref| / rms(ref) and the figure the tolerance applies to (which, for
    outputs stored in bf16, allows their own rounding 2^-8 |ref| on top)."""
    mod = sys.modules.get("tests.gpu_util")
    rows = getattr(mod, "MARGINS", None) if mod else None
    if not rows:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity margins: output raw/adjusted max err / rms(oracle)")
    by = {}
    for label, key, raw, adj in rows:
        cur = by.setdefault(label, {})
        r0, a0 = cur.get(key, (0.0, 0.0))
        cur[key] = (max(r0, raw), max(a0, adj))
    for label, outs in by.items():
        tr.write_line(f"{label}: " + " ".join(f"{k} {r:.2e}/{a:.2e}" for k, (r, a) in outs.items()))


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)

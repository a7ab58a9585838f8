import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) when no GPU is visible, so that
    # `-m "not gpu"` and plain runs on CPU-only hosts stay green.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU visible")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # How many GEMV outputs were more than one bf16 ulp from RNE(y_ref) (each
    # inside the fp32 bound; see tests/w4_testutil.check_gemv).
    try:
        from tests import w4_testutil as tu
    except Exception:
        return
    if not tu.OFF_ULP_STATS:
        return
    off = sum(o for _, o, _ in tu.OFF_ULP_STATS)
    total = sum(n for _, _, n in tu.OFF_ULP_STATS)
    worst = max(tu.OFF_ULP_STATS, key=lambda t: t[1] / max(t[2], 1))
    terminalreporter.write_line(
        f"bf16 outputs more than 1 ulp from RNE(y_ref): {off} of {total} compared "
        f"in {len(tu.OFF_ULP_STATS)} GEMV checks (largest share: {worst[1]} of {worst[2]} "
        f"in {worst[0]})")

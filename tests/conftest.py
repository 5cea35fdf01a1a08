import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large inputs; minutes of CPU or GPU time")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Reports the drift curves of the chained-step diagnostics and how many
    gated (fused) output elements passed only through the one-bf16-ulp branch
    of their tolerance, per test."""
    parity = sys.modules.get("tests.parity")
    tr = terminalreporter
    for name, curve in sorted(getattr(parity, "DRIFT", {}).items()):
        tr.write_sep("-", f"drift vs the float64 oracle: {name}")
        for step, e_out, e_st in curve:
            tr.write_line(f"step {step:4d}: out max abs {e_out:.3e}, state max abs {e_st:.3e}")
    rows = getattr(parity, "ULP_BRANCH", None)
    if not rows:
        return
    tr.write_sep("-", "gated outputs passing only within one bf16 ulp (error > 2e-3)")
    tot_u = tot_a = 0
    worst = 0.0
    for test, (n_u, n_a, w) in sorted(rows.items()):
        tot_u, tot_a, worst = tot_u + n_u, tot_a + n_a, max(worst, w)
        if n_u:
            tr.write_line(f"{test}: {n_u} of {n_a} elements, worst {w:.2f} half-ulps")
    tr.write_line(f"all tests: {tot_u} of {tot_a} gated output elements used the ulp branch; "
                  f"worst error {worst:.2f} half-ulps")

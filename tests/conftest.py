import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(autouse=True)
def _parity_test_name(request):
    """Tags the parity log entries (tests/helpers.py:max_err) with the running test."""
    import helpers
    helpers.CURRENT_TEST = request.node.nodeid
    yield


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity report: per test, the plain max abs error against the oracle, the error as the bar
    judges it (bf16-resolution allowance above |ref| >= 2), and how many elements needed that
    allowance."""
    try:
        import helpers
    except ImportError:
        return
    if not helpers.PARITY_LOG:
        return
    rows = {}
    for name, plain, judged, used, n in helpers.PARITY_LOG:
        r = rows.setdefault(name, [0.0, float("-inf"), 0, 0, 0])
        r[0] = max(r[0], plain)
        r[1] = max(r[1], judged)
        r[2] += used
        r[3] += n
        r[4] += 1
    tr = terminalreporter
    tr.section("parity report (max abs error vs the fp64 oracle)")
    tr.write_line(f"{'test [compared with]':<104} {'plain':>9} {'judged':>9} {'allow':>6} {'elements':>11}")
    for name, (plain, judged, used, n, calls) in rows.items():
        tr.write_line(f"{name[-104:]:<104} {plain:9.2e} {judged:9.2e} {used:6d} {n:11d}")
    ours = {k: v for k, v in rows.items() if k.endswith("[oracle]")}
    tot_used = sum(r[2] for r in ours.values())
    tot_n = sum(r[3] for r in ours.values())
    worst = max(ours.items(), key=lambda kv: kv[1][0]) if ours else None
    tr.write_line(f"results against the oracle on the same pool: {len(ours)} checks, largest plain max abs error "
                  f"{worst[1][0]:.3e} ({worst[0]}); elements over the plain 1e-2 bar brought under it by the "
                  f"bf16-resolution allowance: {tot_used} of {tot_n}" if worst else "no checks against the oracle")

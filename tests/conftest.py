import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels through the C ABI)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Sum of the GPU parity counts (tests/gpu_util.compare) over the
    session, and the tests that saw near-boundary decisions."""
    try:
        import gpu_util
    except Exception:  # noqa: BLE001 -- CPU-only sessions never import it
        return
    log = gpu_util.PARITY_LOG
    if not log:
        return
    keys = ("requests", "exact", "near_accept", "near_draw", "draw_mismatch", "path_mismatch")
    tot = {k: sum(st[k] for _, st in log) for k in keys}
    worst = max(st["max_mismatch_margin"] for _, st in log)
    tr = terminalreporter
    tr.write_sep("-", "GPU parity against the oracle")
    tr.write_line(f"comparisons {len(log)}; " + ", ".join(f"{k} {tot[k]}" for k in keys) +
                  f"; largest oracle margin of a mismatching draw {worst:.3g}")
    if tot["requests"]:
        tr.write_line(f"near draws {tot['near_draw'] / tot['requests']:.3%} of requests, "
                      f"near accept tests on {tot['near_accept']} requests")
    for name, st in log:
        if st["near_accept"] or st["near_draw"]:
            tr.write_line(f"  {name}: " + ", ".join(f"{k} {st[k]}" for k in keys[1:]))

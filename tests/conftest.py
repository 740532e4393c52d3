import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels through the C ABI)")


def pytest_collection_modifyitems(config, items):
    """A gpu-marked test on a machine without a GPU is a skip, never a pass."""
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


# ---- parity report: elements that pass only through the half-ulp term ----
#
# The parity rule is |gpu - ref| <= tol * sum|w*x| + 1e-6 + half_ulp(ref); the
# last term admits the output cast's own rounding.  Every check goes through
# oracle.violations, which counts the elements that would fail without that
# term; this records the count per test and prints the totals at the end.

_ROUNDING_REPORT = []


@pytest.fixture(autouse=True)
def _rounding_only_count(request):
    import oracle
    before = dict(oracle.ROUNDING_ONLY)
    yield
    n = oracle.ROUNDING_ONLY["elements"] - before["elements"]
    m = oracle.ROUNDING_ONLY["checked"] - before["checked"]
    if m:
        request.node.user_properties.append(("rounding_only_elements", n))
        request.node.user_properties.append(("checked_elements", m))
        _ROUNDING_REPORT.append((request.node.nodeid, n, m))


def pytest_terminal_summary(terminalreporter):
    if not _ROUNDING_REPORT:
        return
    tot_n = sum(r[1] for r in _ROUNDING_REPORT)
    tot_m = sum(r[2] for r in _ROUNDING_REPORT)
    tr = terminalreporter
    tr.write_sep("-", "parity: elements passing only through the half-ulp rounding term")
    for nodeid, n, m in _ROUNDING_REPORT:
        if n or "test_full_size_workload" in nodeid:
            tr.write_line(f"{n:>10} of {m:>12}  {nodeid}")
    tr.write_line(f"{tot_n:>10} of {tot_m:>12}  all {len(_ROUNDING_REPORT)} checking tests")

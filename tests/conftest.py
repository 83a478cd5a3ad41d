import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


# Stochastic decisions the parity tests excused because the oracle's uniform
# lay within the tolerance of a decision boundary: (test, excused, compared).
BOUNDARY_CASES = []


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def golden():
    import json

    def load(name):
        with open(os.path.join(ROOT, "tests", "golden", name)) as f:
            return json.load(f)
    return load


@pytest.fixture(scope="session")
def boundary_report():
    """Record (label, excused, compared) for the terminal summary."""
    def add(label, excused, compared):
        BOUNDARY_CASES.append((label, int(excused), int(compared)))
    return add


@pytest.fixture(autouse=True)
def _debug_bounds(request):
    """Under the bounds-checking build (SPECDEC_DEBUG=1) every GPU test ends
    with no out-of-range index met by any kernel it launched."""
    if os.environ.get("SPECDEC_DEBUG") != "1" or request.node.get_closest_marker("gpu") is None:
        yield
        return
    import speculative_decoding_draft_select_gb300 as sd
    assert sd.library_path.endswith("libspecdec_debug.so")
    sd.spec_debug_bounds(reset=True)
    yield
    n = sd.spec_debug_bounds(reset=True)
    assert n == 0, f"{n} out-of-range indices met under the bounds-checking build"


def pytest_terminal_summary(terminalreporter):
    if not BOUNDARY_CASES:
        return
    tr = terminalreporter
    total = sum(e for _, e, _ in BOUNDARY_CASES)
    tr.write_sep("-", f"boundary-excused stochastic decisions: {total}")
    for label, excused, compared in BOUNDARY_CASES:
        tr.write_line(f"{label}: {excused} of {compared} requests differ only within 1e-5 of a decision boundary")

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Decisions compared bit for bit, and those left out because the oracle's own
# decision sat inside a margin, per parity test (reported, not hidden).
_MARGINS = {}


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def golden():
    def load(name):
        with open(os.path.join(GOLDEN, name)) as f:
            return json.load(f)
    return load


@pytest.fixture
def margins(request, record_property):
    """margins(compared, near): record how many decisions a parity test compared
    bit for bit and how many it skipped as near-margin.  They go into the junit
    properties, the terminal summary and, when SPEC_MARGINS_JSON names a file,
    that file."""
    def rec(compared, near):
        _MARGINS[request.node.nodeid] = {"compared": int(compared), "near_margin": int(near)}
        record_property("compared", int(compared))
        record_property("near_margin", int(near))
    return rec


def pytest_terminal_summary(terminalreporter):
    if not _MARGINS:
        return
    terminalreporter.write_sep("-", "decisions compared / near-margin (skipped) per parity test")
    for k, v in sorted(_MARGINS.items()):
        terminalreporter.write_line(f"{k}: compared {v['compared']}, near-margin {v['near_margin']}")
    out = os.environ.get("SPEC_MARGINS_JSON")
    if out:
        with open(out, "w") as f:
            json.dump(_MARGINS, f, indent=1, sort_keys=True)

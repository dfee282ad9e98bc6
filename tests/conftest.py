import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libgdn")
    config.addinivalue_line("markers", "slow: long CPU test")


def read_golden(name):
    """Parse a golden text fixture: 'key v1 v2 ...' per line, '#' comments."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            vals = []
            for p in parts[1:]:
                try:
                    vals.append(float(p))
                except ValueError:
                    vals.append(p)
            out[parts[0]] = vals
    return out


@pytest.fixture
def golden():
    return read_golden


@pytest.fixture(autouse=True)
def _canaries(request, monkeypatch):
    """GPU tests: guard bands around every buffer a libgdn call writes."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import guards
    guards.install(monkeypatch)
    yield


def pytest_terminal_summary(terminalreporter):
    """The o error yardsticks over every GPU comparison of the run (see
    gpu_harness.REPORT): the largest of each, relative to rms(o_ref)."""
    tr = terminalreporter
    g = sys.modules.get("guards")
    if g and g.checked["calls"]:
        tr.write_sep("-", "canaries: %d guarded calls, %d buffers, every guard band intact"
                     % (g.checked["calls"], g.checked["buffers"]))
    h = sys.modules.get("gpu_harness")
    rep = getattr(h, "REPORT", None) if h else None
    if not rep:
        return
    tr.write_sep("-", "o error over %d comparisons (max, relative to rms(o_ref))" % len(rep))
    for key, label in (("excess", "asserted: |o_gpu - o_ref| - bf16 quantum"),
                       ("plain", "plain: |o_gpu - o_ref|"),
                       ("rne", "against bf16_rne(o_ref): |o_gpu - rne(o_ref)|"),
                       ("rne_ulps", "the same in bf16 ulps, where |o_ref| >= rms/16")):
        vals = [r[key] for r in rep if key in r]
        if vals:
            tr.write_line("  %-52s %.3e" % (label, max(vals)))

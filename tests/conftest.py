import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libskv.so")


def pytest_terminal_summary(terminalreporter):
    """The largest errors the GPU parity tests measured against the oracle."""
    h = sys.modules.get("gpu_harness")
    if h is None or not getattr(h, "MEASURED", None):
        return
    tr = terminalreporter
    tr.section("measured errors against the fp64 oracle (largest per test)")
    for test, rec in sorted(h.MEASURED.items()):
        tr.write_line("%-60s %s" % (test[:60], "  ".join("%s %.3g" % kv for kv in sorted(rec.items()))))

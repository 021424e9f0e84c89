import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libcsa.so")


def _observed_errors():
    mod = sys.modules.get("tests.parity_helpers")
    return list(getattr(mod, "ERRORS", [])) if mod is not None else []


def pytest_terminal_summary(terminalreporter):
    """The largest error of each checked quantity over the session; with
    CSA_PARITY_LOG set, every recorded (test, quantity, error) as JSON there."""
    errs = _observed_errors()
    if not errs:
        return
    worst = {}
    for test, what, e in errs:
        if what not in worst or e > worst[what][0]:
            worst[what] = (e, test)
    terminalreporter.write_line("observed parity errors (largest per quantity):")
    for what in sorted(worst):
        e, test = worst[what]
        terminalreporter.write_line(f"  {what:34s} {e:.6g}  ({test})")
    path = os.environ.get("CSA_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            json.dump([{"test": t, "quantity": w, "error": e} for t, w, e in errs], f, indent=0)

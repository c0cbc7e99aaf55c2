import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    import json
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def pytest_terminal_summary(terminalreporter):
    """The parity margins the GPU tests recorded: worst err / row RMS of each
    check beside its bound."""
    mod = sys.modules.get("gpu_util")
    margins = getattr(mod, "MARGINS", None) if mod else None
    if not margins:
        return
    terminalreporter.write_sep("-", "parity margins: max over rows of err / row RMS (bound)")
    for test, label, err, tol in margins:
        terminalreporter.write_line(f"{err:10.3e}  (bound {tol:.0e})  {test}  {label}")

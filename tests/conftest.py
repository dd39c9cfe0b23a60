import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libs5.so")
    config.addinivalue_line("markers", "slow: full-size parity case")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints every parity check of the session: rel-L2 and max-abs error
    against the oracle (or the path named), with the tolerance applied."""
    mod = sys.modules.get("_parity")
    log = getattr(mod, "PARITY_LOG", None) if mod else None
    if not log:
        return
    tr = terminalreporter
    tr.section("parity (rel-L2 / max-abs error per check)")
    tr.write_line("%-72s %-26s %10s %10s %10s %8s" % ("test", "quantity", "rel-L2", "max-abs", "max|ref|", "tol"))
    for test, what, r, m, scale, tol in log:
        name = test if len(test) <= 72 else "..." + test[-69:]
        tr.write_line("%-72s %-26s %10.3e %10.3e %10.3e %8.1e" % (name, what[:26], r, m, scale, tol))
    path = os.environ.get("S5_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            for row in log:
                f.write("\t".join(str(v) for v in row) + "\n")

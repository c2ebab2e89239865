import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# (case, max-abs, rel-L2, bound) of every parity comparison made in this session; printed at the
# end so a run's log records how far each case sits from the tolerance, not only that it passed.
MARGINS: list[tuple[str, float, float, str]] = []


def record_margin(case: str, max_abs: float, rel_l2: float, bound: str = "4e-3 / 1e-2") -> None:
    MARGINS.append((case, float(max_abs), float(rel_l2), bound))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if not MARGINS:
        return
    tr = terminalreporter
    tr.write_sep("-", f"parity margins ({len(MARGINS)} comparisons; bound = max-abs / rel-L2)")
    worst = max(MARGINS, key=lambda m: m[1])
    for case, err, rl2, bound in MARGINS:
        tr.write_line(f"{case:64s} max-abs {err:.3e}  rel-L2 {rl2:.3e}  bound {bound}")
    tr.write_line(f"largest max-abs: {worst[1]:.3e} ({worst[0]})")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    import torch

    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity comparisons of the session: raw max-abs next to the bound, and how many entries
    passed only through the half-ulp allowance for bf16 outputs (tests/parity.py)."""
    try:
        from tests.parity import MAX_ABS, RECORDS
    except Exception:  # pragma: no cover - the module failed to import; nothing recorded
        return
    if not RECORDS:
        return
    tr = terminalreporter
    n_allow = sum(r[4] for r in RECORDS)
    n_tot = sum(r[5] for r in RECORDS)
    worst = sorted(RECORDS, key=lambda r: -r[2])[:8]
    tr.write_sep("-", f"parity: {len(RECORDS)} comparisons, {n_allow} of {n_tot} entries above "
                      f"max-abs {MAX_ABS} raw (all within half a bf16 ulp of it)")
    for name, rel, raw, beyond, na, n in worst:
        tr.write_line(f"  {name:12s} rel L2 {rel:.2e}  raw max abs {raw:.2e}  beyond ulp "
                      f"{beyond:.2e}  needed allowance {na}/{n}")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Routing exclusions of the GPU parity checks, one line per checked layer: tokens whose
    k-th and (k+1)-th oracle logits are within 1e-5 (excluded from the bit-exact id check)
    and slot-order swaps between selected experts whose logits are within 1e-5."""
    parity = sys.modules.get("parity")
    recs = getattr(parity, "EXCLUSIONS", None) if parity else None
    if not recs:
        return
    tr = terminalreporter
    tr.write_sep("-", "routing exclusions of the parity checks (near ties < 1e-5)")
    n_near = sum(len(r["near_ties"]) for r in recs)
    n_swap = sum(len(r["order_ties"]) for r in recs)
    for r in recs:
        extra = ""
        if "experts_compared_fully" in r:
            extra = f"; experts compared on every row {r['expert_rows']}"
        tr.write_line(f"{r['name']}: near-tie tokens {r['near_ties']}, slot-order swaps {r['order_ties']} "
                      f"(bound {r['bound']} each); y rows compared {r.get('y_rows_compared', '-')}, "
                      f"tokens compared {r.get('tokens_compared', '-')}{extra}")
    tr.write_line(f"total: {len(recs)} layers checked, {n_near} near-tie tokens excluded, {n_swap} slot-order swaps")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (full-size workloads)")
    # mutation test: plant one mistake in the oracle before the pin tests
    # are collected (set only by test_oracle_mutants.py in a child process)
    name = os.environ.get("ORACLE_MUTANT")
    if name:
        import _oracle_mutants
        _oracle_mutants.apply(name)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Per-tensor error of the floating-point parity checks: plain
    max|err|/RMS(ref) and the checked quantity (the error beyond half a
    bf16 step, over RMS), the largest first."""
    try:
        import _helpers
    except ImportError:
        return
    recs = _helpers.RECORDS
    if not recs:
        return
    tr = terminalreporter
    tr.section("parity error per tensor (max|err|/RMS, bound 2e-2 after half a bf16 step)")
    worst = sorted(recs, key=lambda r: -r[2])
    tr.write_line(f"{len(recs)} comparisons; largest checked excess/RMS {worst[0][2]:.3e} "
                  f"({worst[0][0]}); largest plain max|err|/RMS "
                  f"{max(r[1] for r in recs):.3e}")
    for name, plain, exc in worst[:25]:
        tr.write_line(f"  {exc:10.3e}  {plain:10.3e}  {name}")

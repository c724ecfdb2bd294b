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

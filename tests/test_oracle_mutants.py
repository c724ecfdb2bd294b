"""Mutation test of the oracle's pins: every planted mistake in
``_oracle_mutants.MUTANTS`` must make at least one pin test fail.

The pins are the CPU tests that tie the oracle to what the pages and the
mathematics fix (worked routing examples, closed forms, brute force on tiny
inputs, finite differences, exact special cases, invariants).  Each mutant
runs them in a child pytest process with ORACLE_MUTANT set; ``conftest.py``
plants the mistake in the oracle before collection.  A mutant whose child
run passes is a mistake no pin would catch, and fails this test.  The
unmutated oracle must pass the same run (checked first), so a kill is the
mutant's doing."""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

import _oracle_mutants as MUT

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PINS = ["test_oracle_mlp.py", "test_oracle_mx.py", "test_oracle_mx_bwd.py",
        "test_oracle_routing.py"]


def _run(mutant):
    env = dict(os.environ)
    env.pop("ORACLE_MUTANT", None)
    if mutant:
        env["ORACLE_MUTANT"] = mutant
    env.setdefault("OMP_NUM_THREADS", "1")
    env.setdefault("OPENBLAS_NUM_THREADS", "1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
           "-m", "not gpu", *[os.path.join(HERE, p) for p in PINS]]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return mutant, r.returncode, r.stdout[-2000:]


def test_every_planted_mistake_fails_a_pin():
    name, rc, out = _run(None)
    assert rc == 0, f"the unmutated oracle fails its pins:\n{out}"
    workers = max(1, min(8, os.cpu_count() or 1))
    survivors, broken = [], []
    with cf.ThreadPoolExecutor(workers) as ex:
        for mutant, rc, out in ex.map(_run, list(MUT.MUTANTS)):
            if rc == 0:
                survivors.append(mutant)
            elif rc != 1:                  # 1 = tests failed; anything else = no run
                broken.append((mutant, rc, out))
    assert not broken, f"mutants that did not run: {broken}"
    assert not survivors, f"planted mistakes no pin catches: {survivors}"

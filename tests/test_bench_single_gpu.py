"""The bench runs on one GPU only: its grouped GEMMs use cluster-multicast
TMA loads, which are kept to single-GPU processes.  Under torchrun with
WORLD_SIZE > 1, or with --gpus > 1, it prints one "unavailable" line on
rank 0 and exits with status 2 before any CUDA or process-group call
(checked here on the CPU)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=env,
                          capture_output=True, text=True, timeout=300)


def test_world_size_two_is_refused_on_rank0():
    r = _run(["--gpus", "2"], {"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode == 2, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert "unavailable" in j and "single-GPU" in j["unavailable"]


def test_other_ranks_print_nothing():
    r = _run(["--gpus", "2"], {"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 2 and r.stdout.strip() == ""


def test_gpus_flag_alone_is_refused():
    r = _run(["--gpus", "4"], {"WORLD_SIZE": "1"})
    assert r.returncode == 2
    assert "unavailable" in json.loads(r.stdout.strip())

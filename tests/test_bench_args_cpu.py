"""bench.py's single-workload modes reject malformed shapes before touching the GPU
(the argument is parsed first), and its help lists every mode."""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=300)


@pytest.mark.parametrize("args, message", [
    (["--forward", "1,2,3"], "--forward wants B,H,N,d,causal"),
    (["--forward", "1,2,3,4,5,6,7"], "--forward wants B,H,N,d,causal"),
    (["--forward", "1,2,128,64,0,-1"], "--forward wants B,H,N,d,causal"),
    (["--forward", "a,b,c,d,e"], "--forward wants B,H,N,d,causal"),
    (["--backward", "1,2,3"], "--backward wants B,H,N,d,causal"),
    (["--rows", "columns"], "--rows wants state or softmax"),
])
def test_malformed_mode_arguments_exit_with_a_message(args, message):
    r = _bench(*args, "--steps", "1", "--warmup", "3")
    assert r.returncode != 0
    assert message in r.stderr


def test_warmup_below_three_is_refused():
    r = _bench("--warmup", "2")
    assert r.returncode != 0 and "--warmup must be at least 3" in r.stderr


def test_help_lists_every_mode():
    r = _bench("--help")
    assert r.returncode == 0
    for flag in ("--suite", "--backward", "--forward", "--rows", "--impl", "--gpus"):
        assert flag in r.stdout

"""Calls from several host threads at once, each on its own stream, from a
cold start (a fresh process), checked against the oracle: the library's
host-side caches and first-use set-up are shared across threads."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_concurrent_host_threads_from_a_cold_start():
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([HERE, os.path.dirname(HERE), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, os.path.join(HERE, "threads_child.py")], capture_output=True, text=True,
                       timeout=600, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count(" 0 wrong") == 6, r.stdout

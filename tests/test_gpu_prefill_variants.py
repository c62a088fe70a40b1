"""GPU parity of both prefill kernels whatever the shape: the 128 x 256 tile
kernel forced on small and ragged problems (the library picks it by tile
count, so the default tests reach it only at full size), and the 128 x 128
kernel forced at the full-size M = 4096 problem.  Each runs in a child
process because the library reads PQ2_PREFILL_WIDE once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(mode, names):
    env = dict(os.environ, PQ2_PREFILL_WIDE=mode, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "prefill_variant_child.py"),
                        *names], env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    for n in names:
        assert f"ok {n}" in r.stdout, r.stdout


def test_wide_kernel_on_small_and_ragged_shapes():
    _run("1", ["ragged", "m17", "m300", "m129", "n512"])


def test_narrow_kernel_at_full_size():
    _run("2", ["m4096"])

"""The int8 / int4 tcgen05 tile's parity cases (tests/tcq_cases.py), run in a
child pytest whose DG_TUNE=TQ=8 routes every int8 / int4 launch of 8+ tokens
to that tile: the library reads DG_TUNE once per process, and by default it
sends only long int4 rows there."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tcgen05_int_tile_cases_in_a_child_process():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, DG_TUNE="TQ=8")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(HERE, "tcq_cases.py")], cwd=os.path.dirname(HERE), env=env,
                       capture_output=True, text=True, timeout=900)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    summary = [l for l in r.stdout.splitlines() if l.strip()][-1]
    assert " passed" in summary and "skipped" not in summary and "failed" not in summary, tail

"""The fp16 / bf16 tcgen05 tile's stream-K split under forced grids
(tests/tc_grid_cases.py), each grid in a child pytest whose DG_TUNE=TG=g
sets it: the library reads DG_TUNE once per process."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("grid", [5, 37, 151, 256])
def test_tcgen05_tile_under_a_forced_grid_in_a_child_process(grid):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, DG_TUNE="TG=%d" % grid)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(HERE, "tc_grid_cases.py")], cwd=os.path.dirname(HERE), env=env,
                       capture_output=True, text=True, timeout=900)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    summary = [l for l in r.stdout.splitlines() if l.strip()][-1]
    assert " passed" in summary and "skipped" not in summary and "failed" not in summary, tail

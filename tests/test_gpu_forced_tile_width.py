"""Tile widths that only the FP8FG_BN override selects: 192 columns (never
chosen automatically) and 128 columns for problems of more than one row
block. The override is read once per process, so each width runs in a child
process (forced_tile_width_case.py) that checks its results against the
oracle and exits non-zero on a mismatch."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("bn", [128, 192])
def test_forced_tile_width_matches_oracle(bn):
    env = dict(os.environ, FP8FG_BN=str(bn))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "forced_tile_width_case.py")], env=env,
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout + r.stderr)[-4000:]
    assert f"tile width {bn}: ok" in r.stdout

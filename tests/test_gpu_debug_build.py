"""The debug build (-DMLA_DEBUG: every global store, query load, tile
coordinate and combine index checked against its buffer, a failed check
reported as MLA_DERR_DEBUG_BOUNDS instead of made) runs every kernel variant
without a failed check and with the release build's parity."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_reports_no_out_of_bounds_access():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_build_check.py")],
                       capture_output=True, text=True, timeout=1800, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    results = json.loads(r.stdout.strip().splitlines()[-1])
    assert len(results) == 21
    for name, st in results.items():
        assert st["err"] == 0, (name, st)
        assert st["finite"] and st["violations"] == 0 and st["rel_l2"] <= 1e-2, (name, st)

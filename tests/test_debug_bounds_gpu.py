"""The checked-index build (VH_DEBUG_BOUNDS) on small and ragged shapes.

``compute-sanitizer`` is closed on the GPU pool, so the scan kernels carry their own
bounds checks in a debug build of the library (libvh_dbg.so): every global access
computed from an index (pixels along a route, the scan's slices of memories0,
memories_out and the backward records, the readout adds) and the shared-memory rows
addressed by token position are checked before they are made; a failed check is counted
in stats[VH_STAT_BOUNDS] and the access skipped.  Each case runs in a child process that
loads that library, and must count no failed check and match the oracle."""
import json
import os
import subprocess
import sys

import pytest

from tests._helpers import TOL

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_counts_no_failed_check():
    from visual_backbone_gb300 import _build
    _build.build(debug=True)
    env = dict(os.environ, VH_DEBUG_BOUNDS="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_debug_bounds_cases.py")],
                         env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    rows = [json.loads(l) for l in res.stdout.splitlines() if l.startswith("{")]
    from tests._debug_bounds_cases import CASES
    assert [r["name"] for r in rows] == [c[0] for c in CASES]
    for r in rows:
        assert r["bounds"] == 0 and r["timeout"] == 0, r
        assert r["err"] < TOL, r

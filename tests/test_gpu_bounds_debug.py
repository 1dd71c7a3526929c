"""The bounds-checked build of the library (TROP_DEBUG_BOUNDS=1) on the GPU: built here, then
driven through every stage of the path in a process of its own (tests/bounds_cases.py, with
TROP_LIBRARY=debug so that the package loads it).  Every case must match the oracle and the
library must have recorded no access outside a tensor's byte range.  No case provokes a
violation of a real tensor: the inputs are the ordinary parity inputs; the one control case
narrows every checked range by 4 bytes (a test hook) so that a permute's last element counts as
outside, and the record must then show it.  The access is skipped, not made, and the element
lies inside the tensor's memory in any case."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def debug_lib():
    from einsum_device_side_gb300 import build
    return build.build(variant="debug")


def test_debug_build_every_stage_in_bounds_and_exact(debug_lib):
    env = dict(os.environ, TROP_LIBRARY="debug")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bounds_cases.py")], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["library"] == debug_lib
    assert res["cases"] >= 60
    assert res["failures"] == [], res["failures"]
    rep = res["report"]
    assert rep is not None, "the debug library did not answer the bounds report"
    assert rep["count"] == 0, f"out-of-range accesses: {rep}"
    ctl = res["control"]
    assert ctl is not None and ctl["count"] >= 1 and ctl["file"] == "unary.cu", ctl

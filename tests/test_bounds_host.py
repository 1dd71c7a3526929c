"""Host checks of the bounds-checked debug build: the byte-range arithmetic of csrc/bounds.h
(compiled with g++ against a stand-in record, no GPU), and the normal build's answer to the
report call (TROP_ERR_UNSUPPORTED: it checks nothing)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "einsum_device_side_gb300", "csrc")


def _cuda_include():
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        inc = os.path.join(cand, "include")
        if cand and os.path.exists(os.path.join(inc, "cuda_runtime.h")):
            return inc
    return None


def test_span_arithmetic(tmp_path):
    cxx = shutil.which("g++")
    inc = _cuda_include()
    if not cxx or not inc:
        pytest.skip("g++ or the CUDA headers are missing")
    exe = str(tmp_path / "bounds_span_check")
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-DTROP_DEBUG_BOUNDS=1", "-I", CSRC, "-I", inc,
                        os.path.join(ROOT, "tests", "bounds_span_check.cpp"), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout


def test_normal_build_reports_unsupported():
    from einsum_device_side_gb300 import build
    build.build()
    import einsum_device_side_gb300 as t
    t.load()
    assert t.debug_bounds_report() is None
    assert t.debug_bounds_trim(4) is False

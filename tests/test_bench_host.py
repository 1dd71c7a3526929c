"""Host-side checks of bench.py's bookkeeping (no GPU): the DRAM-traffic record it reports is
keyed to the GEMM source's code, so edits to comments keep it and edits to code drop it."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sha(tmp_path, text):
    p = tmp_path / "k.cu"
    p.write_text(text)
    return bench.code_sha256(str(p))


def test_code_hash_ignores_comments_and_whitespace(tmp_path):
    base = _sha(tmp_path, "int f(int a) {\n    return a + 1;  // add one\n}\n")
    assert _sha(tmp_path, "int f(int a)\n{\n  /* a note */ return a + 1;\n}\n") == base
    assert _sha(tmp_path, "// header\nint f(int a) { return a + 1; }\n") == base


def test_code_hash_sees_code_and_string_literals(tmp_path):
    base = _sha(tmp_path, 'const char* s = "x"; int f(int a) { return a + 1; }\n')
    assert _sha(tmp_path, 'const char* s = "x"; int f(int a) { return a + 2; }\n') != base
    assert _sha(tmp_path, 'const char* s = "y"; int f(int a) { return a + 1; }\n') != base
    # comment markers inside a string literal are code, not comments
    assert _sha(tmp_path, 'const char* s = "// x"; int f(int a) { return a + 1; }\n') != base


def test_traffic_record_parses():
    f = os.path.join(ROOT, "profiles", "k_gemm_tma_fused_traffic.txt")
    kv = dict(line.split(": ", 1) for line in open(f).read().splitlines() if ": " in line)
    assert int(kv["bytes_per_launch"]) > 0 and len(kv["source_code_sha256"]) == 64


def test_traffic_record_matches_the_current_gemm_source():
    """The committed traffic record belongs to gemm.cu as it stands (bench.py then reports it)."""
    assert bench.gemm_traffic() is not None


def test_cpu_baseline_on_one_thread_reports_one_core():
    r = bench.cpu_sample_rate(target_s=0.3, threads=1)
    assert r["cores"] == 1 and r["kind"] == "oracle" and r["value"] > 0
    assert "1 thread" in r["sample"]

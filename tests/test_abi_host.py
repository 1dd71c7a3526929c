"""Host-side checks of the C-ABI library: it loads, exports every entry point
include/tropical.h declares, and its planner (pure host logic) lowers specs
as intended.  No GPU and no compute call."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def trop():
    from einsum_device_side_gb300 import build
    build.build()
    import einsum_device_side_gb300 as t
    t.load()
    return t


def _declared():
    txt = open(os.path.join(ROOT, "include", "tropical.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(tropical_[a-z0-9_]+)\s*\(", txt)))


def test_header_declares_the_path_entry_points():
    names = _declared()
    for need in ("tropical_permute_trace", "tropical_gemm_strided_batched_argmax", "tropical_einsum_pairwise",
                 "tropical_contract_tree", "tropical_init", "tropical_sync_pool", "tropical_stats",
                 "tropical_last_error"):
        assert need in names


def test_library_exports_every_declared_symbol(trop):
    lib = ctypes.CDLL(trop.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_stats_without_gpu(trop):
    assert trop.version() == 2
    s = trop.stats()
    assert s["stream_syncs"] == 0


def _desc(spec, sa, sb):
    import numpy as np
    st = lambda shp: list(np.cumprod([1] + list(shp[::-1]))[:-1][::-1])  # noqa: E731
    return st(sa), st(sb)


@pytest.mark.parametrize("spec,sa,sb,expect", [
    ("bmk,bkn->bmn", [64, 256, 256], [64, 256, 256], "gemm M=256 N=256 K=256 batch_axes=1"),
    ("zacd,zdce->zea", [16, 512, 32, 32], [16, 32, 32, 512], "permB gemm M=512 N=512 K=1024"),
    ("ij,jk->k", [4, 6], [6, 5], "reduceA gemm M=1 N=5 K=6"),
    ("iij,jk->ik", [5, 5, 7], [7, 4], "gemm M=5 N=4 K=7"),
    ("alub,lun->alnb", [8, 2, 2, 16], [2, 2, 2], "gemm M=16 N=2 K=2 batch_axes=2"),
    ("ln,un->lun", [2, 2], [2, 2], "gemm M=2 N=2 K=1 batch_axes=1"),
])
def test_planner_lowering(trop, spec, sa, sb, expect):
    st_a, st_b = _desc(spec, sa, sb)
    text = trop.plan_describe(spec, sa, st_a, sb, st_b)
    assert text.startswith(expect), text


def test_planner_transposed_output_is_staged_not_permuted(trop):
    # the planner does not permute for a transposed output; the GEMM dispatcher
    # writes the tiled product to a contiguous buffer and transposes it once
    st_a, st_b = _desc("bmk,bkn->bnm", [2, 64, 32], [2, 32, 48])
    text = trop.plan_describe("bmk,bkn->bnm", [2, 64, 32], st_a, [2, 32, 48], st_b)
    assert "perm" not in text and "sCm=1" in text and "route=tiled staged" in text


@pytest.mark.parametrize("spec,sa,sb,route", [
    ("bmk,bkn->bmn", [64, 256, 256], [64, 256, 256], "route=tiled"),
    ("alub,lun->alnb", [8, 2, 2, 16], [2, 2, 2], "route=stream"),
    ("ij,jk->ik", [5, 300], [300, 7], "route=generic"),
])
def test_planner_reports_the_gemm_route(trop, spec, sa, sb, route):
    st_a, st_b = _desc(spec, sa, sb)
    text = trop.plan_describe(spec, sa, st_a, sb, st_b)
    assert route in text, text


@pytest.mark.parametrize("spec,err", [
    ("ij,jk->q", "SPEC"), ("ij,jk", "SPEC"), ("i1,jk->ik", "SPEC"), ("ij,jk->ii", "SPEC"),
])
def test_planner_rejects_bad_specs(trop, spec, err):
    with pytest.raises(trop.TropicalError) as e:
        trop.plan_describe(spec, [2, 3], [3, 1], [3, 4], [4, 1])
    assert e.value.name == err


def test_planner_rejects_inconsistent_extents(trop):
    with pytest.raises(trop.TropicalError) as e:
        trop.plan_describe("ij,jk->ik", [2, 3], [3, 1], [4, 5], [5, 1])
    assert e.value.name == "SHAPE"


def _contig(shape):
    st, acc = [], 1
    for d in reversed(shape):
        st.append(acc)
        acc *= d
    return list(reversed(st))


@pytest.mark.parametrize("k, kernel, resolve", [(256, "tma", "fused"), (64, "tma", "fused"), (16, "tma", "fused"),
                                                (512, "tma", "panel32"), (1024, "tma", "panel16"),
                                                (40, "tiled", "rows"), (72, "tiled", "rows"),
                                                (257, "tiled", "panel64")])
def test_describe_names_gemm_kernel_and_resolve(trop, k, kernel, resolve):
    """The planner reports which argmax GEMM kernel and resolve pass a layout takes: the TMA-fed
    kernel needs one batch axis, K a multiple of 16 and 16-byte row strides; the row resolve
    needs K <= 256 in whole chunks of 8, and after the TMA-fed kernel it runs in the same launch
    ("fused").  Batch 64 of 128 x 128 tiles fills more than half a
    wave, so no tile is split along k (a split tail takes the cp.async kernel)."""
    sa, sb = [64, 128, k], [64, k, 128]
    text = trop.plan_describe("zmk,zkn->zmn", sa, _contig(sa), sb, _contig(sb))
    assert f"kernel={kernel}" in text and f"resolve={resolve}" in text, text


def test_describe_small_problems_split_the_tail_on_the_cpasync_kernel(trop):
    """Under half a wave of tiles the argmax GEMM cuts its tiles along k (stream-K), which
    only the cp.async kernel does: the planner says so instead of naming the TMA kernel."""
    sa, sb = [8, 128, 256], [8, 256, 128]
    text = trop.plan_describe("zmk,zkn->zmn", sa, _contig(sa), sb, _contig(sb))
    assert "split_tail" in text and "kernel=tiled" in text, text


def test_describe_tma_needs_aligned_rows_and_one_batch_axis(trop):
    # rows of A 16 floats + 1 apart: not 16-byte aligned, so the cp.async kernel
    text = trop.plan_describe("zmk,zkn->zmn", [4, 64, 16], [64 * 17, 17, 1], [4, 16, 64], [1024, 64, 1])
    assert "kernel=tiled" in text, text
    # two batch axes that do not merge into one: the cp.async kernel
    sa, sb = [3, 5, 64, 32], [3, 5, 32, 64]
    st_a = [5 * 64 * 32 + 64, 64 * 32, 32, 1]
    text = trop.plan_describe("yzmk,yzkn->yzmn", sa, st_a, sb, _contig(sb))
    assert "kernel=tiled" in text and "batch_axes=2" in text, text


def test_describe_wide_row_strides_leave_the_32_bit_paths(trop):
    """A row stride past 2^31 elements keeps the GEMM on 64-bit offsets: the short-K row resolve
    (32-bit row offsets, in its own launch or fused with the TMA-fed GEMM) gives way to the
    64-bit panel resolve, at any M."""
    wide = (1 << 31) + 64
    sb = [1, 64, 128]
    narrow = trop.plan_describe("zmk,zkn->zmn", [1, 16, 64], [16 * 64, 64, 1], sb, _contig(sb))
    assert "route=tiled" in narrow and ("resolve=rows" in narrow or "resolve=fused" in narrow), narrow
    text = trop.plan_describe("zmk,zkn->zmn", [1, 16, 64], [16 * wide, wide, 1], sb, _contig(sb))
    assert "route=tiled" in text and "resolve=panel64" in text, text
    assert f"sAm={wide}" in text, text


def test_fastcall_binding_loads_and_marshals(trop):
    """The CPython binding of the hot entry points is built beside the library and reaches
    the same C ABI: wrong argument counts raise, and an unknown semiring comes back as the
    library's INVALID_ARG code before any device work."""
    import sysconfig
    if not os.path.exists(os.path.join(sysconfig.get_paths()["include"], "Python.h")):
        pytest.skip("no Python headers: the ctypes binding serves every call")
    fc = trop._fc
    assert fc is not None
    with pytest.raises(TypeError):
        fc.gemm(1, 2)
    rc = fc.permute_trace(None, 0, (2, 3), (3, 1), b"ij->ji", 7, None, 0, (3, 2), (2, 1), None, None, False)
    assert rc == -1 and "semiring" in fc.last_error()
    rc = fc.gemm(7, 0, 1, 2, 2, 2, None, 0, 0, 0, None, 0, 0, 0, None, 0, 0, 0, None, None)
    assert rc == -1
    with pytest.raises(ValueError):
        fc.permute_trace(None, 0, (1,) * 33, (1,) * 33, b"a->a", 0, None, 0, (1,), (1,), None, None, False)

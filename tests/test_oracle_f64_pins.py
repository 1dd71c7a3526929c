"""Pins of the oracle's binary64 path: hand-computed products, a pure-Python
brute force on tiny inputs (Python floats are IEEE binary64, each + or * rounds
once), a case only binary64 resolves, and numpy references for the unary path."""

import itertools
import json
import os

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("sr", [0, 1, 2])
def test_f64_hand_products(sr):
    """Every hand-computed case of tests/golden/hand_products.json, in binary64."""
    g = json.load(open(os.path.join(ROOT, "golden", "hand_products.json")))
    name = ["maxplus", "minplus", "maxtimes"][sr]
    n = 0
    for case in g["cases"]:
        if name not in case:
            continue
        a = np.array(case["A"], dtype=np.float64)[None]
        b = np.array(case["B"], dtype=np.float64)[None]
        c, i = oracle.gemm(a, b, sr)
        np.testing.assert_array_equal(c[0], np.array(case[name]["C"], dtype=np.float64))
        np.testing.assert_array_equal(i[0], np.array(case[name]["I"]))
        n += 1
    assert n >= 1


def _brute(spec_a, spec_b, spec_o, a, b, sr):
    sizes = {}
    for l, s in zip(spec_a, a.shape):
        sizes[l] = s
    for l, s in zip(spec_b, b.shape):
        sizes[l] = s
    k_labels = [l for l in dict.fromkeys(spec_a) if l in spec_b and l not in spec_o]
    r_labels = [l for l in dict.fromkeys(spec_a + spec_b) if l not in spec_o and l not in k_labels]
    zero = {0: -np.inf, 1: np.inf, 2: 0.0}[sr]
    better = (lambda t, u: t < u) if sr == 1 else (lambda t, u: t > u)
    out = np.empty([sizes[l] for l in spec_o])
    arg = np.empty(out.shape, dtype=np.int32)
    for oi in itertools.product(*[range(sizes[l]) for l in spec_o]):
        best, idx = zero, 0
        for kn, kv in enumerate(itertools.product(*[range(sizes[l]) for l in k_labels])):
            v = zero
            for rv in itertools.product(*[range(sizes[l]) for l in r_labels]):
                val = dict(zip(spec_o, oi)) | dict(zip(k_labels, kv)) | dict(zip(r_labels, rv))
                x = float(a[tuple(val[l] for l in spec_a)])
                y = float(b[tuple(val[l] for l in spec_b)])
                p = x * y if sr == 2 else x + y
                if better(p, v):
                    v = p
            if better(v, best):
                best, idx = v, kn
        out[oi] = best
        arg[oi] = idx
    return out, arg


@pytest.mark.parametrize("sr", [0, 1, 2])
@pytest.mark.parametrize("spec", ["ij,jk->ik", "bij,bjk->bki", "ijk,jkl->li", "ij,jk->k"])
def test_f64_pairwise_matches_python_brute_force(sr, spec):
    ops, out = spec.split("->")
    la, lb = ops.split(",")
    rng = np.random.default_rng(len(spec) + sr)
    sizes = {ch: int(rng.integers(1, 4)) for ch in set(la + lb)}
    lo = 0.0 if sr == 2 else -1.0
    a = rng.uniform(lo, 1.0, [sizes[c] for c in la])
    b = rng.uniform(lo, 1.0, [sizes[c] for c in lb])
    got, garg = oracle.einsum(spec, a, b, semiring=sr)
    want, warg = _brute(la, lb, out, a, b, sr)
    assert got.dtype == np.float64
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(garg, warg)


def test_f64_keeps_what_f32_rounds_away():
    a = np.array([[[1.0 + 2.0 ** -30, 0.0]]])
    b = np.array([[[1.0], [1.0 + 2.0 ** -31]]])
    c, i = oracle.gemm(a, b, 0)
    assert c[0, 0, 0] == 2.0 + 2.0 ** -30 and i[0, 0, 0] == 0     # both sums differ only beyond binary32
    c32, _ = oracle.gemm(a.astype(np.float32), b.astype(np.float32), 0)
    assert float(c32[0, 0, 0]) == 2.0


def test_f64_unary_permute_and_trace():
    x = synth.uniform_f32(5, (3, 4, 5, 2), -1, 1).astype(np.float64) * (1 + 2.0 ** -40)
    y, _ = oracle.einsum("abcd->dbca", x)
    np.testing.assert_array_equal(y, np.transpose(x, (3, 1, 2, 0)))
    t = synth.uniform_f32(6, (6, 6, 3), -1, 1).astype(np.float64) * (1 + 2.0 ** -40)
    d, da = oracle.einsum("iij->j", t, semiring=0)
    diag = np.diagonal(t, axis1=0, axis2=1)          # (j, i)
    np.testing.assert_array_equal(d, diag.max(axis=1))
    np.testing.assert_array_equal(da, diag.argmax(axis=1))

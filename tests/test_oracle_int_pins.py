"""Pins for the oracle's integer contractions (i32 and i64 operands).

Reading: each tropical product is the exact integer a + b (a * b for max-times),
the inputs must make every product fit the operand type, and the semiring
zero is the type's min / max / 0 (it starts the running (+); it is never an
operand value).  The pages name integer types for the permute/gather and the
argmax but fix no overflow policy for integer contractions; this is the
plainest reading that keeps results exact.

These tests tie the integer branch of the oracle to Python's unbounded
integers (brute force over every label assignment), to hand computations, to
Floyd-Warshall, to the already pinned binary32 branch on values every type
holds exactly, and check that a product outside the type is refused.  No GPU.
"""

import itertools
import json
import os

import numpy as np
import pytest

import oracle
from oracle import MAXPLUS, MINPLUS, MAXTIMES

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NAMES = {"maxplus": MAXPLUS, "minplus": MINPLUS, "maxtimes": MAXTIMES}
INTS = (np.int32, np.int64)


def _zero(sr, dt):
    if sr == MAXTIMES:
        return 0
    info = np.iinfo(dt)
    return info.min if sr == MAXPLUS else info.max


def _brute_int(la, lb, lo, a, b, sr):
    """Every full label assignment, products in Python integers (exact); value = (+) of the
    terms of an output index, argmax = smallest contracted linear index (labels in
    first-appearance order in the first operand) with a term equal to the value, 0 when
    nothing beats the zero."""
    sizes = dict(zip(la, a.shape))
    sizes.update(zip(lb, b.shape))
    labels = sorted(sizes)
    kl = [l for l in dict.fromkeys(la) if l in lb and l not in lo]
    zero = _zero(sr, a.dtype)
    better = (lambda x, y: x < y) if sr == MINPLUS else (lambda x, y: x > y)
    best, arg = {}, {}
    for vals in itertools.product(*[range(sizes[l]) for l in labels]):
        v = dict(zip(labels, vals))
        x = int(a[tuple(v[l] for l in la)])
        y = int(b[tuple(v[l] for l in lb)])
        t = x * y if sr == MAXTIMES else x + y
        o = tuple(v[l] for l in lo)
        k = 0
        for l in kl:
            k = k * sizes[l] + v[l]
        cur = best.get(o, zero)
        if better(t, cur) or (t == cur and o in arg and k < arg[o] and t != zero):
            best[o], arg[o] = t, k
    shape = tuple(sizes[l] for l in lo)
    c = np.full(shape, zero, dtype=a.dtype)
    i = np.zeros(shape, dtype=np.int32)
    for o, t in best.items():
        c[o] = t
        i[o] = arg[o]
    return c, i


def test_hand_products_in_both_integer_types():
    with open(os.path.join(GOLDEN, "hand_products.json")) as f:
        data = json.load(f)
    n = 0
    for dt in INTS:
        for case in data["cases"]:
            a = np.array(case["A"], dtype=dt)[None]
            b = np.array(case["B"], dtype=dt)[None]
            for name, sr in NAMES.items():
                if name not in case:
                    continue
                c, i = oracle.gemm(a, b, sr)
                assert c.dtype == dt
                np.testing.assert_array_equal(c[0], np.array(case[name]["C"], dtype=dt), err_msg=case["name"])
                np.testing.assert_array_equal(i[0], np.array(case[name]["I"], dtype=np.int32), err_msg=case["name"])
                n += 1
    assert n == 18


def _random_pair_case(rng):
    pool = "abcde"
    sizes = {l: int(rng.integers(1, 4)) for l in pool}
    if rng.random() < 0.1:
        sizes[pool[int(rng.integers(0, 5))]] = 0
    la = [pool[int(rng.integers(0, 5))] for _ in range(int(rng.integers(1, 5)))]
    lb = [pool[int(rng.integers(0, 5))] for _ in range(int(rng.integers(1, 4)))]
    present = list(dict.fromkeys(la + lb))
    lo = [l for l in present if rng.random() < 0.5]
    rng.shuffle(lo)
    return la, lb, lo, sizes


@pytest.mark.parametrize("dt", INTS)
@pytest.mark.parametrize("scale", ["ties", "wide"])
def test_integer_einsum_against_exact_brute_force(dt, scale):
    """Random tiny specs (repeated labels, one-operand labels, zero extents).  'ties': values in
    [-4, 4] (many equal terms: the argmax must take the smallest index); 'wide': values near
    the type's range (i32: |v| < 2^29, beyond binary32's 24 bits; i64: |v| < 2^61, beyond
    binary64's 53 bits), so a float shortcut anywhere would round."""
    rng = np.random.default_rng(11 + (dt == np.int64) + 2 * (scale == "wide"))
    for trial in range(150):
        la, lb, lo, sizes = _random_pair_case(rng)
        sr = int(rng.integers(0, 3))
        if scale == "ties":
            lo_v, hi_v = (0, 4) if sr == MAXTIMES else (-4, 4)
        elif sr == MAXTIMES:
            hi_v = (1 << 15) if dt == np.int32 else (1 << 31)   # products stay inside the type
            lo_v = 0
        else:
            hi_v = (1 << 29) if dt == np.int32 else (1 << 61)
            lo_v = -hi_v
        a = rng.integers(lo_v, hi_v + 1, size=[sizes[l] for l in la], dtype=np.int64).astype(dt)
        b = rng.integers(lo_v, hi_v + 1, size=[sizes[l] for l in lb], dtype=np.int64).astype(dt)
        spec = (list(map(ord, la)), list(map(ord, lb)), list(map(ord, lo)))
        c, i = oracle.einsum(spec, a, b, sr)
        rc, ri = _brute_int(spec[0], spec[1], spec[2], a, b, sr)
        np.testing.assert_array_equal(c, rc, err_msg=f"{la},{lb}->{lo} sr={sr}")
        np.testing.assert_array_equal(i, ri, err_msg=f"{la},{lb}->{lo} sr={sr}")


@pytest.mark.parametrize("dt", INTS)
def test_integer_branch_equals_the_binary32_branch_on_small_values(dt):
    """Values that binary32 holds exactly (and whose products it holds exactly): the integer
    and the (separately pinned) binary32 definitions must give the same values and argmax."""
    rng = np.random.default_rng(21)
    for sr in (MAXPLUS, MINPLUS, MAXTIMES):
        lo_v = 0 if sr == MAXTIMES else -1000
        a = rng.integers(lo_v, 1001, size=(3, 17, 23)).astype(dt)
        b = rng.integers(lo_v, 1001, size=(3, 23, 19)).astype(dt)
        c, i = oracle.gemm(a, b, sr)
        cf, i_f = oracle.gemm(a.astype(np.float32), b.astype(np.float32), sr)
        np.testing.assert_array_equal(c, cf.astype(dt))
        np.testing.assert_array_equal(i, i_f)


def test_minplus_powers_are_floyd_warshall_in_integers():
    from scipy.sparse.csgraph import floyd_warshall
    rng = np.random.default_rng(31)
    n = 10
    w = rng.integers(1, 1000, size=(n, n)).astype(np.int64)
    np.fill_diagonal(w, 0)
    for dt in INTS:
        d = w.astype(dt)[None]
        for _ in range(4):      # paths of up to 16 edges >= n - 1
            d, _ = oracle.gemm(d, d, MINPLUS)
        ref = floyd_warshall(w.astype(np.float64), directed=True)
        np.testing.assert_array_equal(d[0], ref.astype(dt))


def test_exact_beyond_binary64():
    """i64 max-plus and max-times whose results binary64 cannot hold: exact."""
    a = np.array([[[(1 << 62) - 7, 3]]], dtype=np.int64)              # 1 x 1 x 2
    b = np.array([[[5], [1]]], dtype=np.int64)                         # 1 x 2 x 1
    c, i = oracle.gemm(a, b, MAXPLUS)
    assert int(c[0, 0, 0]) == (1 << 62) - 2 and int(i[0, 0, 0]) == 0
    a = np.array([[[3037000493, 7]]], dtype=np.int64)
    b = np.array([[[3037000493], [1]]], dtype=np.int64)
    c, i = oracle.gemm(a, b, MAXTIMES)
    assert int(c[0, 0, 0]) == 3037000493 * 3037000493 and int(i[0, 0, 0]) == 0


@pytest.mark.parametrize("dt,big", [(np.int32, 1 << 30), (np.int64, 1 << 62)])
def test_a_product_outside_the_type_is_refused(dt, big):
    a = np.array([[[big, 0]]], dtype=dt)
    b = np.array([[[big], [1]]], dtype=dt)
    with pytest.raises(OverflowError):
        oracle.gemm(a, b, MAXPLUS)
    with pytest.raises(OverflowError):
        oracle.gemm(-a, -b - 1, MINPLUS)       # -2^k + (-2^k - 1) is one below the type's minimum
    # the same operands with the offending product never formed are fine
    c, _ = oracle.gemm(a[:, :, 1:], b[:, 1:, :], MAXPLUS)
    assert int(c[0, 0, 0]) == 1


def test_integer_argmax_certificate_and_strict_ties():
    rng = np.random.default_rng(41)
    for dt in INTS:
        a = rng.integers(-3, 4, size=(2, 9, 31)).astype(dt)
        b = rng.integers(-3, 4, size=(2, 31, 8)).astype(dt)
        c, i = oracle.gemm(a, b, MAXPLUS)
        t = a.astype(np.int64)[:, :, :, None] + b.astype(np.int64)[:, None, :, :]
        np.testing.assert_array_equal(c, t.max(axis=2))
        np.testing.assert_array_equal(i, t.argmax(axis=2))       # numpy: the first maximum
        assert ((t == c[:, :, None, :].astype(np.int64)).sum(axis=2) > 1).mean() > 0.3   # ties are common

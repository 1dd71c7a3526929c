"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties the oracle to a hand computation, a library routine, brute-force
enumeration, a closed form or an algebraic invariant, chosen so that a dropped
term, a wrong sign or index, a transposed operand or a wrong tie rule fails at
least one of them.  No GPU, no CUDA library.
"""

import itertools
import json
import os

import numpy as np
import pytest

import oracle
import synth
from oracle import MAXPLUS, MINPLUS, MAXTIMES

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ZERO = {MAXPLUS: -np.inf, MINPLUS: np.inf, MAXTIMES: 0.0}
NAMES = {"maxplus": MAXPLUS, "minplus": MINPLUS, "maxtimes": MAXTIMES}


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# hand computations (tests/golden/hand_products.json)

def test_hand_products():
    with open(os.path.join(GOLDEN, "hand_products.json")) as f:
        data = json.load(f)
    n = 0
    for case in data["cases"]:
        a = np.array(case["A"], dtype=np.float32)[None]
        b = np.array(case["B"], dtype=np.float32)[None]
        for name, sr in NAMES.items():
            if name not in case:
                continue
            c, i = oracle.gemm(a, b, sr)
            np.testing.assert_array_equal(c[0], np.array(case[name]["C"], dtype=np.float32), err_msg=f"{case['name']} {name}")
            np.testing.assert_array_equal(i[0], np.array(case[name]["I"], dtype=np.int32), err_msg=f"{case['name']} {name}")
            n += 1
    assert n == 9


# --------------------------------------------------------------------------
# special cases that reduce to textbook results

def test_identity_matrices():
    rng = _rng(1)
    a = rng.integers(-5, 6, size=(1, 5, 7)).astype(np.float32)
    for sr, one, zero in ((MAXPLUS, 0.0, -np.inf), (MINPLUS, 0.0, np.inf)):
        eye = np.full((1, 7, 7), zero, dtype=np.float32)
        eye[0, np.arange(7), np.arange(7)] = one
        c, i = oracle.gemm(a, eye, sr)            # A (x) I = A, winner k = n
        np.testing.assert_array_equal(c, a)
        np.testing.assert_array_equal(i[0], np.tile(np.arange(7), (5, 1)))
        eye5 = np.full((1, 5, 5), zero, dtype=np.float32)
        eye5[0, np.arange(5), np.arange(5)] = one
        c, i = oracle.gemm(eye5, a, sr)           # I (x) A = A, winner k = m
        np.testing.assert_array_equal(c, a)
        np.testing.assert_array_equal(i[0], np.tile(np.arange(5)[:, None], (1, 7)))
    ap = np.abs(a) + 1
    eye = np.zeros((1, 7, 7), dtype=np.float32)
    eye[0, np.arange(7), np.arange(7)] = 1.0
    c, i = oracle.gemm(ap, eye, MAXTIMES)
    np.testing.assert_array_equal(c, ap)
    np.testing.assert_array_equal(i[0], np.tile(np.arange(7), (5, 1)))


def test_k1_is_outer_product():
    rng = _rng(2)
    a = rng.uniform(0.1, 1, size=(2, 6, 1)).astype(np.float32)
    b = rng.uniform(0.1, 1, size=(2, 1, 5)).astype(np.float32)
    for sr in (MAXPLUS, MINPLUS, MAXTIMES):
        c, i = oracle.gemm(a, b, sr)
        ref = a * b if sr == MAXTIMES else a + b
        np.testing.assert_array_equal(c, ref)
        assert (i == 0).all()


def test_minplus_powers_are_floyd_warshall():
    from scipy.sparse.csgraph import floyd_warshall
    rng = _rng(3)
    n = 9
    w = rng.integers(1, 20, size=(n, n)).astype(np.float64)
    mask = rng.random((n, n)) < 0.35
    w[mask] = np.inf
    np.fill_diagonal(w, 0.0)
    d = w.astype(np.float32)[None]
    for _ in range(4):  # paths of up to 16 edges >= n-1
        d, _ = oracle.gemm(d, d, MINPLUS)
    ref = floyd_warshall(np.where(np.isinf(w), 0, w), directed=True)
    np.testing.assert_array_equal(d[0], ref.astype(np.float32))


def test_gemm_matches_numpy_broadcast_and_first_argmax():
    rng = _rng(4)
    for sr in (MAXPLUS, MINPLUS, MAXTIMES):
        lo = 0.0 if sr == MAXTIMES else -1.0
        a = rng.uniform(lo, 1, size=(3, 7, 11)).astype(np.float32)
        b = rng.uniform(lo, 1, size=(3, 11, 5)).astype(np.float32)
        t = a[:, :, :, None] * b[:, None, :, :] if sr == MAXTIMES else a[:, :, :, None] + b[:, None, :, :]
        assert t.dtype == np.float32
        if sr == MINPLUS:
            ref_c, ref_i = t.min(axis=2), t.argmin(axis=2)
        else:
            ref_c, ref_i = t.max(axis=2), t.argmax(axis=2)   # numpy: first occurrence
        c, i = oracle.gemm(a, b, sr)
        np.testing.assert_array_equal(c, ref_c)
        np.testing.assert_array_equal(i, ref_i)


def test_ties_from_integer_inputs_break_to_smallest_k():
    a, b = synth.gemm64_inputs()
    c, i = oracle.gemm(a, b, MAXPLUS)
    t = a[:, :, :, None] + b[:, None, :, :]
    np.testing.assert_array_equal(c, t.max(axis=2))
    np.testing.assert_array_equal(i, t.argmax(axis=2))
    # the workload really has ties: several k reach the maximum for a quarter of outputs
    assert ((t == c[:, :, None, :]).sum(axis=2) > 1).mean() > 0.2


def test_strided_views_and_broadcast_batch():
    rng = _rng(5)
    base = rng.uniform(-1, 1, size=(4, 9, 12)).astype(np.float32)
    a = base[:, 1:8:2, ::3]                  # non-contiguous
    bb = rng.uniform(-1, 1, size=(1, 4, 6)).astype(np.float32)
    b = np.broadcast_to(bb, (4, 4, 6))       # batch stride 0
    c, i = oracle.gemm(a, b, MAXPLUS)
    c2, i2 = oracle.gemm(np.ascontiguousarray(a), np.ascontiguousarray(b), MAXPLUS)
    np.testing.assert_array_equal(c, c2)
    np.testing.assert_array_equal(i, i2)
    t = a[:, :, :, None] + b[:, None, :, :]
    np.testing.assert_array_equal(c, t.max(axis=2))


# --------------------------------------------------------------------------
# brute force on tiny random specs

def _brute(la, lb, lo, a, b, sr):
    """Enumerate every full label assignment; value = (+) of all terms grouped
    by output index; argmax = smallest contracted linear index (labels in
    first-appearance order in the first operand) having some term equal to the
    value, or 0 when nothing beats the semiring zero."""
    sizes = {}
    for l, s in zip(la, a.shape):
        sizes[l] = s
    if b is not None:
        for l, s in zip(lb, b.shape):
            sizes[l] = s
    labels = sorted(sizes)
    pairwise = b is not None
    if pairwise:
        kl = [l for l in dict.fromkeys(la) if l in lb and l not in lo]
    else:
        kl = [l for l in dict.fromkeys(la) if l not in lo]
    out_shape = tuple(sizes[l] for l in lo)
    terms = {}
    for vals in itertools.product(*[range(sizes[l]) for l in labels]):
        v = dict(zip(labels, vals))
        x = a[tuple(v[l] for l in la)]
        if pairwise:
            y = b[tuple(v[l] for l in lb)]
            t = np.float32(x * y) if sr == MAXTIMES else np.float32(x + y)
        else:
            t = x
        o = tuple(v[l] for l in lo)
        k = 0
        for l in kl:
            k = k * sizes[l] + v[l]
        terms.setdefault(o, []).append((t, k))
    dt = a.dtype
    if dt == np.float32:
        zero = np.float32(ZERO[sr])
    elif sr == MAXTIMES:
        zero = dt.type(0)
    else:
        info = np.iinfo(dt)
        zero = dt.type(info.min if sr == MAXPLUS else info.max)
    c = np.full(out_shape, zero, dtype=dt)
    arg = np.zeros(out_shape, dtype=np.int32)
    for o, lst in terms.items():
        vals = [t for t, _ in lst]
        best = min(vals) if sr == MINPLUS else max(vals)
        beats = (best < zero) if sr == MINPLUS else (best > zero)
        if beats:
            c[o] = best
            arg[o] = min(k for t, k in lst if t == best)
    return c, arg


def _random_case(rng, pairwise):
    pool = "abcde"
    sizes = {l: int(rng.integers(1, 4)) for l in pool}
    if rng.random() < 0.1:
        sizes[pool[int(rng.integers(0, 5))]] = 0
    la = [pool[int(rng.integers(0, 5))] for _ in range(int(rng.integers(1, 5)))]
    lb = [pool[int(rng.integers(0, 5))] for _ in range(int(rng.integers(1, 4)))] if pairwise else []
    present = list(dict.fromkeys(la + lb))
    lo = [l for l in present if rng.random() < 0.5]
    rng.shuffle(lo)
    return la, (lb if pairwise else None), lo, sizes


@pytest.mark.parametrize("pairwise", [False, True])
def test_einsum_against_brute_force(pairwise):
    rng = _rng(6 + pairwise)
    for trial in range(120):
        la, lb, lo, sizes = _random_case(rng, pairwise)
        sr = int(rng.integers(0, 3))
        lo_v = 0.0 if sr == MAXTIMES else -4.0
        if pairwise or rng.random() < 0.5:
            dt = np.float32
            a = np.round(rng.uniform(lo_v, 4, size=[sizes[l] for l in la])).astype(np.float32)
        else:
            dt = np.int32 if rng.random() < 0.5 else np.int64
            a = rng.integers(-5 if sr != MAXTIMES else 0, 6, size=[sizes[l] for l in la]).astype(dt)
        b = None
        if pairwise:
            b = np.round(rng.uniform(lo_v, 4, size=[sizes[l] for l in lb])).astype(np.float32)
        spec = (list(map(ord, la)), list(map(ord, lb)) if lb is not None else None, list(map(ord, lo)))
        c, i = oracle.einsum(spec, a, b, sr)
        rc, ri = _brute(spec[0], spec[1], spec[2], a, b, sr)
        np.testing.assert_array_equal(c, rc, err_msg=f"{la},{lb}->{lo} sr={sr}")
        np.testing.assert_array_equal(i, ri, err_msg=f"{la},{lb}->{lo} sr={sr}")


# --------------------------------------------------------------------------
# permute / diagonal / trace

@pytest.mark.parametrize("dtype", [np.float32, np.int32, np.int64])
def test_permute_matches_numpy_and_inverts(dtype):
    rng = _rng(8)
    x = (rng.uniform(-100, 100, size=(3, 4, 2, 5, 3)) * 7).astype(dtype)
    perm = [3, 0, 4, 2, 1]
    src = "abcde"
    dst = "".join(src[p] for p in perm)
    y, i = oracle.einsum(f"{src}->{dst}", x)
    np.testing.assert_array_equal(y, np.transpose(x, perm))
    assert (i == 0).all()
    inv = list(np.argsort(perm))
    z, _ = oracle.einsum(f"{dst}->{src}", y)
    assert z.tobytes() == x.tobytes()
    del inv


def test_diagonal_and_trace_match_numpy():
    x = synth.uniform_f32(123, (6, 6, 4, 5), -1, 1)
    d, i = oracle.einsum("iijk->ijk", x)
    ref = np.stack([x[n, n] for n in range(6)])
    np.testing.assert_array_equal(d, ref)
    assert (i == 0).all()
    for sr, fn, afn in ((MAXPLUS, np.max, np.argmax), (MINPLUS, np.min, np.argmin)):
        t, ti = oracle.einsum("iijk->jk", x, semiring=sr)
        np.testing.assert_array_equal(t, fn(ref, axis=0))
        np.testing.assert_array_equal(ti, afn(ref, axis=0))
    # full reduction with argmax over two labels, row-major in first appearance
    t, ti = oracle.einsum("ijk->", x[0], semiring=MAXPLUS)
    assert t == x[0].max() and ti == int(np.argmax(x[0]))
    # label absent from the output and repeated: 'iij->j' reduces the diagonal
    t, ti = oracle.einsum("iij->j", x[:, :, 0, :], semiring=MAXPLUS)
    diag = np.stack([x[n, n, 0] for n in range(6)])
    np.testing.assert_array_equal(t, diag.max(axis=0))
    np.testing.assert_array_equal(ti, diag.argmax(axis=0))


def test_trace_then_contract_equals_contract_then_trace():
    rng = _rng(9)
    a = rng.uniform(-1, 1, size=(5, 5, 7)).astype(np.float32)
    b = rng.uniform(-1, 1, size=(7, 4)).astype(np.float32)
    direct, di = oracle.einsum("iij,jk->ik", a, b)
    d1, _ = oracle.einsum("iij->ij", a)
    r1, ri1 = oracle.einsum("ij,jk->ik", d1, b)
    full, fi = oracle.einsum("aij,jk->aik", a, b)
    r2, ri2 = oracle.einsum("iik->ik", full)
    ri2b = np.stack([fi[n, n] for n in range(5)])
    for r, ri in ((r1, ri1), (r2, ri2b)):
        np.testing.assert_array_equal(direct, r)
        np.testing.assert_array_equal(di, ri)
    assert (ri2 == 0).all()


def test_one_operand_labels_fold_before_argmax():
    """'ij,jk->k': i only in A is reduced first; argmax indexes j alone."""
    rng = _rng(10)
    a = rng.integers(-3, 4, size=(4, 6)).astype(np.float32)
    b = rng.integers(-3, 4, size=(6, 5)).astype(np.float32)
    c, i = oracle.einsum("ij,jk->k", a, b)
    amax = a.max(axis=0)
    t = amax[:, None] + b
    np.testing.assert_array_equal(c, t.max(axis=0))
    np.testing.assert_array_equal(i, t.argmax(axis=0))


def test_semirings_differ_and_are_not_standard_algebra():
    a, b = synth.gemm_batched_inputs(2, batch=1, m=8, n=8, k=8)
    res = [oracle.gemm(a, b, sr)[0] for sr in (MAXPLUS, MINPLUS, MAXTIMES)]
    std = np.matmul(a, b)
    for x in range(3):
        assert not np.array_equal(res[x], std)
        for y in range(x):
            assert not np.array_equal(res[x], res[y])


def test_argmax_certifies_value():
    a, b = synth.gemm_batched_inputs(0, batch=2, m=16, n=16, k=33)
    c, i = oracle.gemm(a, b, MAXPLUS)
    for bb in range(2):
        for m in range(16):
            for n in range(16):
                t = a[bb, m, :] + b[bb, :, n]
                k = i[bb, m, n]
                assert t[k] == c[bb, m, n]
                assert (t[:k] < c[bb, m, n]).all() and (t <= c[bb, m, n]).all()


def test_empty_contraction_and_empty_output():
    a = np.zeros((2, 3, 0), dtype=np.float32)
    b = np.zeros((2, 0, 4), dtype=np.float32)
    for sr in (MAXPLUS, MINPLUS, MAXTIMES):
        c, i = oracle.gemm(a, b, sr)
        assert c.shape == (2, 3, 4)
        assert (c == np.float32(ZERO[sr])).all() and (i == 0).all()
    c, i = oracle.gemm(np.zeros((2, 0, 5), np.float32), np.zeros((2, 5, 4), np.float32))
    assert c.shape == (2, 0, 4) and i.shape == (2, 0, 4)


def test_samples_equal_full_evaluation():
    a, b = synth.gemm_batched_inputs(1, batch=2, m=9, n=10, k=13)
    c, i = oracle.gemm(a, b, MINPLUS)
    s = np.array([0, 5, 17, 179, 99, 3], dtype=np.int64)
    cs, is_ = oracle.gemm(a, b, MINPLUS, samples=s)
    np.testing.assert_array_equal(cs, c.reshape(-1)[s])
    np.testing.assert_array_equal(is_, i.reshape(-1)[s])


# --------------------------------------------------------------------------
# spin glass

@pytest.mark.parametrize("rows,cols,seed", [(2, 2, 1), (2, 3, 2), (3, 3, 3), (3, 4, 4), (2, 7, 5), (4, 4, 6), (4, 5, 7)])
def test_ising_elimination_equals_brute_force(rows, cols, seed):
    jh, jv = synth.couplings(seed, rows, cols)
    w, spins = oracle.ising_ground(jh, jv, rows, cols, nthreads=1)
    wb, sb = oracle.ising_brute(jh, jv, rows, cols)
    assert w == wb
    assert oracle.ising_energy(jh, jv, spins) == -w
    assert oracle.ising_energy(jh, jv, sb) == -wb


def test_ising_workload_4x4_instance():
    jh, jv = synth.ising_couplings(4, 4)
    w, spins = oracle.ising_ground(jh, jv, 4, 4)
    wb, _ = oracle.ising_brute(jh, jv, 4, 4)
    assert w == wb and oracle.ising_energy(jh, jv, spins) == -w


@pytest.mark.parametrize("sign", [1, -1])
def test_ising_uniform_couplings_closed_form(sign):
    rows, cols = 10, 12
    jh = np.full((rows, cols - 1), sign, np.int8)
    jv = np.full((rows - 1, cols), sign, np.int8)
    nbonds = rows * (cols - 1) + (rows - 1) * cols
    w, spins = oracle.ising_ground(jh, jv, rows, cols)
    assert w == nbonds
    s = spins.astype(int)
    if sign > 0:
        assert (s == s[0, 0]).all()
    else:
        assert (s[:, 1:] == -s[:, :-1]).all() and (s[1:, :] == -s[:-1, :]).all()


def test_ising_backtrack_energy_matches_value_larger_grid():
    jh, jv = synth.couplings(77, 12, 12)
    w, spins = oracle.ising_ground(jh, jv, 12, 12)
    assert oracle.ising_energy(jh, jv, spins) == -w
    assert abs(w) <= 12 * 11 * 2

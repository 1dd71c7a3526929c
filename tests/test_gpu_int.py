"""GPU parity for integer contractions (i32, i64): the strided-batched GEMM with argmax, the
pairwise einsum and a contraction tree, bitwise against the CPU oracle through the C ABI.

Inputs respect the precondition that every product fits the operand type: tie-heavy small
integers, and wide values (i32 |v| < 2^29, beyond binary32's 24 bits; i64 |v| < 2^61, beyond
binary64's 53 bits), so any float shortcut would round."""

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

SR = (0, 1, 2)
INTS = {"i32": np.int32, "i64": np.int64}


@pytest.fixture(scope="module")
def trop():
    import einsum_device_side_gb300 as t
    t.load()
    return t


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _ints(seed, shape, sr, dt, wide):
    if wide:
        hi = ((1 << 15) if dt == np.int32 else (1 << 31)) if sr == 2 else ((1 << 29) if dt == np.int32 else (1 << 61))
    else:
        hi = 4
    lo = 0 if sr == 2 else -hi
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(dt)


def _check(trop, a, b, sr, ad=None, bd=None, **kw):
    ad = _dev(a) if ad is None else ad
    bd = _dev(b) if bd is None else bd
    c, i = trop.gemm(ad, bd, sr, **kw)
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    assert c.dtype == ad.dtype
    assert c.cpu().numpy().tobytes() == np.ascontiguousarray(rc).tobytes()
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


@pytest.mark.parametrize("dt", ["i32", "i64"])
@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("wide", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (3, 70, 45, 37), (2, 130, 129, 70), (1, 64, 64, 64),
                                   (4, 17, 300, 16), (1, 66, 40, 1032)])
def test_int_gemm_matches_oracle(trop, dt, sr, wide, shape):
    bt, m, n, k = shape
    a = _ints(1 + m, (bt, m, k), sr, INTS[dt], wide)
    b = _ints(2 + n, (bt, k, n), sr, INTS[dt], wide)
    _check(trop, a, b, sr)


@pytest.mark.parametrize("dt", ["i32", "i64"])
@pytest.mark.parametrize("layout", ["NT", "TN", "TT"])
def test_int_gemm_transposed_operands_and_output(trop, dt, layout):
    a = _ints(5, (2, 96, 50), 0, INTS[dt], False)
    b = _ints(6, (2, 50, 80), 0, INTS[dt], False)
    ad, bd = _dev(a), _dev(b)
    if layout[0] == "T":
        ad = _dev(np.ascontiguousarray(np.swapaxes(a, 1, 2))).transpose(1, 2)
    if layout[1] == "T":
        bd = _dev(np.ascontiguousarray(np.swapaxes(b, 1, 2))).transpose(1, 2)
    out = torch.empty((2, 80, 96), dtype=ad.dtype, device="cuda").transpose(1, 2)
    am = torch.empty((2, 80, 96), dtype=torch.int32, device="cuda").transpose(1, 2)
    c, i = trop.gemm(ad, bd, 0, out=out, out_argmax=am)
    rc, ri = oracle.gemm(a, b, 0, nthreads=0)
    np.testing.assert_array_equal(c.cpu().numpy(), rc)
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


@pytest.mark.parametrize("dt", ["i32", "i64"])
@pytest.mark.parametrize("sr", SR)
def test_int_gemm_empty_contraction_and_no_argmax(trop, dt, sr):
    t = torch.int32 if dt == "i32" else torch.int64
    c, i = trop.gemm(torch.empty((2, 5, 0), dtype=t, device="cuda"), torch.empty((2, 0, 7), dtype=t, device="cuda"), sr)
    info = np.iinfo(INTS[dt])
    zero = 0 if sr == 2 else (info.min if sr == 0 else info.max)
    assert (c.cpu().numpy() == zero).all() and (i.cpu().numpy() == 0).all()
    a = _ints(7, (2, 33, 20), sr, INTS[dt], True)
    b = _ints(8, (2, 20, 41), sr, INTS[dt], True)
    c = trop.gemm(_dev(a), _dev(b), sr, argmax=False)
    rc, _ = oracle.gemm(a, b, sr, nthreads=0)
    np.testing.assert_array_equal(c.cpu().numpy(), rc)


@pytest.mark.parametrize("sr", SR)
def test_int32_full_size_batched_workload(trop, sr):
    """batch 64 x 256^3 in int32 (entries uniform in [-1000, 1000], [0, 1000] for max-times):
    every output's value and argmax against the oracle."""
    lo = 0 if sr == 2 else -1000
    a = synth.uniform_int(synth.seed_for(synth.W_GEMM_BATCHED, 8 + 2 * sr), (64, 256, 256), lo, 1000, np.int32)
    b = synth.uniform_int(synth.seed_for(synth.W_GEMM_BATCHED, 9 + 2 * sr), (64, 256, 256), lo, 1000, np.int32)
    _check(trop, a, b, sr)


@pytest.mark.parametrize("dt", ["i32", "i64"])
@pytest.mark.parametrize("spec,sa,sb", [
    ("ij,jk->ik", (37, 23), (23, 41)),
    ("ij,jk->ki", (70, 33), (33, 90)),
    ("iij,jk->ik", (9, 9, 7), (7, 5)),            # diagonal in A
    ("ij,jk->k", (6, 8), (8, 5)),                  # one-operand label reduced first
    ("ijk,jkl->li", (5, 6, 7), (6, 7, 4)),
    ("ikj,jkl->il", (5, 7, 6), (6, 7, 4)),         # contracted labels in swapped order: permute
    ("bij,jk->bik", (3, 20, 30), (30, 25)),
    ("zacd,zdce->zea", (2, 5, 3, 4), (2, 4, 3, 6)),
    ("abc,cab->", (3, 4, 5), (5, 3, 4)),
])
@pytest.mark.parametrize("sr", SR)
def test_int_einsum_specs(trop, dt, spec, sa, sb, sr):
    a = _ints(21, sa, sr, INTS[dt], False)
    b = _ints(22, sb, sr, INTS[dt], False)
    o, oa = trop.einsum(spec, _dev(a), _dev(b), sr)
    ro, roa = oracle.einsum(spec, a, b, sr, nthreads=0)
    assert o.cpu().numpy().tobytes() == ro.tobytes(), spec
    np.testing.assert_array_equal(oa.cpu().numpy(), roa, err_msg=spec)


def test_int32_contraction_tree_spin_glass(trop):
    """The 6 x 6 spin glass contracted in int32 (couplings +-1 are exact integers): the tree
    executor's value and back-tracked configuration equal the oracle's elimination."""
    from einsum_device_side_gb300 import ising
    jh, jv = synth.ising_couplings(6, 6)
    inputs, nodes, n_labels, need = ising.build_network(jh, jv)
    dev_inputs = [torch.from_numpy(np.asarray(t).astype(np.int32)).cuda() for t in inputs]
    am = [None] * len(nodes)
    for j in need:
        am[j] = torch.empty([2] * len(nodes[j][4]), dtype=torch.int32, device="cuda")
    out = torch.empty((), dtype=torch.int32, device="cuda")
    trop.contract_tree(dev_inputs, nodes, "maxplus", out, am)
    assign = trop.tree_backtrack(dev_inputs, nodes, am, n_labels, 0)
    w, spins = oracle.ising_ground(jh, jv, 6, 6)
    assert int(out.item()) == w
    np.testing.assert_array_equal(ising.spins_from_assignment(assign.cpu().numpy(), 6, 6), spins)

"""GPU parity in binary64: the f64 GEMM (k_gemm_tiled_f64), f64 reductions,
permutes, pairwise einsum and trees against the CPU oracle, all bit-exact
(values and argmax).  Inputs use the whole 53-bit significand, so a path that
computed in binary32 anywhere would not match.  Calls go through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

SR = (0, 1, 2)


@pytest.fixture(scope="module")
def trop():
    import einsum_device_side_gb300 as t
    t.load()
    return t


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _f64(seed, shape, sr):
    return synth.uniform_f64(seed, shape, 0.0 if sr == 2 else -1.0, 1.0)


def _same(got, ref, what=""):
    assert got.dtype == torch.float64
    assert got.cpu().numpy().tobytes() == np.ascontiguousarray(ref).tobytes(), what


@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 5, 7, 3), (3, 70, 45, 37), (1, 130, 129, 33),
                                   (2, 64, 64, 64), (1, 17, 200, 300), (1, 1, 70, 16)])
def test_gemm_f64_matches_oracle(trop, sr, shape):
    a, b = synth.gemm_batched_inputs(sr, *shape, dtype="f64")
    c, i = trop.gemm(_dev(a), _dev(b), sr)
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    _same(c, rc)
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


@pytest.mark.parametrize("sr", SR)
def test_gemm_f64_full_size_batched_workload(trop, sr):
    """batch 64 x 256^3 in binary64, every output checked."""
    a, b = synth.gemm_batched_inputs(sr, dtype="f64")
    c, i = trop.gemm(_dev(a), _dev(b), sr)
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    _same(c, rc)
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


@pytest.mark.parametrize("sr", SR)
def test_gemm_f64_ties_take_the_smallest_k(trop, sr):
    lo = 0 if sr == 2 else -4
    a = synth.uniform_int(51, (2, 67, 90), lo, 4).astype(np.float64)
    b = synth.uniform_int(52, (2, 90, 71), lo, 4).astype(np.float64)
    c, i = trop.gemm(_dev(a), _dev(b), sr)
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    _same(c, rc)
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


def test_gemm_f64_rounds_in_binary64(trop):
    """1 + 2^-40 survives a binary64 add but not a binary32 one."""
    a = np.array([[[1.0, -3.0]]])
    b = np.array([[[2.0 ** -40], [1.0]]])
    c, i = trop.gemm(_dev(a), _dev(b), "maxplus")
    assert c.item() == 1.0 + 2.0 ** -40 and i.item() == 0


@pytest.mark.parametrize("sr", SR)
def test_gemm_f64_strided_operands_and_transposed_output(trop, sr):
    a, b = synth.gemm_batched_inputs(sr, 2, 48, 40, 150, dtype="f64")
    at = _dev(np.ascontiguousarray(a.transpose(0, 2, 1))).transpose(1, 2)   # sAm = 1
    bt = _dev(np.ascontiguousarray(b.transpose(0, 2, 1))).transpose(1, 2)   # sBk = 1
    out = torch.empty((2, 40, 48), dtype=torch.float64, device="cuda").transpose(1, 2)
    oam = torch.empty((2, 40, 48), dtype=torch.int32, device="cuda").transpose(1, 2)
    c, i = trop.gemm(at, bt, sr, out=out, out_argmax=oam)
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    np.testing.assert_array_equal(c.cpu().numpy(), rc)
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


def test_gemm_f64_empty_extents(trop):
    c, i = trop.gemm(torch.ones((2, 3, 0), dtype=torch.float64, device="cuda"),
                     torch.ones((2, 0, 4), dtype=torch.float64, device="cuda"), "maxplus")
    assert (c.cpu().numpy() == -np.inf).all() and (i.cpu().numpy() == 0).all()
    c, i = trop.gemm(torch.ones((2, 0, 5), dtype=torch.float64, device="cuda"),
                     torch.ones((2, 5, 4), dtype=torch.float64, device="cuda"), "maxplus")
    assert c.shape == (2, 0, 4)


def test_gemm_f64_mixed_dtypes_rejected(trop):
    with pytest.raises(TypeError):
        trop.gemm(torch.ones((1, 2, 2), device="cuda"), torch.ones((1, 2, 2), dtype=torch.float64, device="cuda"))
    with pytest.raises(trop.TropicalError):
        trop.einsum("ij,jk->ik", torch.ones((2, 2), device="cuda"),
                    torch.ones((2, 2), dtype=torch.float64, device="cuda"),
                    out=torch.empty((2, 2), device="cuda"))


@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("spec", ["iijk->ijk", "iijk->jk", "iijk->", "ijkl->li", "iij->i", "ijk->k"])
def test_trace_and_reduce_f64(trop, sr, spec):
    shapes = {"iijk->ijk": (12, 12, 9, 10), "iijk->jk": (12, 12, 9, 10), "iijk->": (12, 12, 9, 10),
              "ijkl->li": (5, 300, 7, 9), "iij->i": (40, 40, 3000), "ijk->k": (300, 5, 70)}
    x = _f64(61, shapes[spec], sr)
    y, am = trop.permute_trace(_dev(x), spec, sr, argmax=True)
    ref, refa = oracle.einsum(spec, x, semiring=sr, nthreads=0)
    _same(y, ref, spec)
    np.testing.assert_array_equal(am.cpu().numpy(), refa)


@pytest.mark.parametrize("sr", SR)
def test_reduce_f64_ties_keep_the_first_index(trop, sr):
    x = synth.uniform_int(62, (300, 5, 70), 0 if sr == 2 else -3, 3).astype(np.float64)
    y, am = trop.permute_trace(_dev(x), "ijk->k", sr, argmax=True)
    ref, refa = oracle.einsum("ijk->k", x, semiring=sr, nthreads=0)
    _same(y, ref)
    np.testing.assert_array_equal(am.cpu().numpy(), refa)


def test_permute_f64(trop):
    x = _f64(63, (16, 16, 16, 16, 16, 16), 0)
    perm = synth.permutation(64, 6)
    spec = "abcdef->" + "".join("abcdef"[p] for p in perm)
    y = trop.permute_trace(_dev(x), spec)
    _same(y, np.transpose(x, perm))


@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("spec,sa,sb", [
    ("zacd,zdce->zea", (2, 64, 8, 8), (2, 8, 8, 72)),
    ("ij,jk->ki", (70, 33), (33, 90)),
    ("iij,jk->ik", (9, 9, 7), (7, 5)),
    ("ij,jk->k", (6, 8), (8, 5)),
    ("ikj,jkl->il", (5, 7, 6), (6, 7, 4)),
    ("bij,jk->bik", (3, 20, 30), (30, 25)),
    ("abc,cab->", (3, 4, 5), (5, 3, 4)),
])
def test_einsum_f64(trop, sr, spec, sa, sb):
    a, b = _f64(71, sa, sr), _f64(72, sb, sr)
    o, oa = trop.einsum(spec, _dev(a), _dev(b), sr)
    ro, roa = oracle.einsum(spec, a, b, sr, nthreads=0)
    _same(o, ro, spec)
    np.testing.assert_array_equal(oa.cpu().numpy(), roa, err_msg=spec)


def test_tree_f64(trop):
    a, b, c = _f64(81, (5, 5, 6), 0), _f64(82, (6, 7), 0), _f64(83, (7, 3), 0)
    I, J, K, L = 0, 1, 2, 3
    nodes = [(0, 1, [I, I, J], [J, K], [K, I]),      # 'iij,jk->ki'
             (3, None, [K, I], None, [I, K]),          # permute 'ki->ik'
             (4, 2, [I, K], [K, L], [I, L])]           # 'ik,kl->il'
    out = torch.empty((5, 3), dtype=torch.float64, device="cuda")
    am = [torch.empty((7, 5), dtype=torch.int32, device="cuda"), None,
          torch.empty((5, 3), dtype=torch.int32, device="cuda")]
    trop.contract_tree([_dev(a), _dev(b), _dev(c)], nodes, "maxplus", out, am)
    r1, ra1 = oracle.einsum("iij,jk->ki", a, b)
    r3, ra3 = oracle.einsum("ik,kl->il", np.ascontiguousarray(r1.T), c)
    _same(out, r3)
    np.testing.assert_array_equal(am[0].cpu().numpy(), ra1)
    np.testing.assert_array_equal(am[2].cpu().numpy(), ra3)

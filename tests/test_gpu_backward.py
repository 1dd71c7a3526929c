"""GPU parity: the tropical GEMM backward (winner routing) vs the CPU oracle.

dA and dB must be bit-identical: both sides add each routed term in the same
order (increasing n for dA, increasing m for dB) with one rounding per
product and per addition.  The argmax fed to both sides is the oracle's, so
this checks the backward alone.  Calls go through tropical_gemm_backward.
"""

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


def _case(sr, batch, m, n, k, seed=0):
    a, b = synth.gemm_batched_inputs(sr, batch=batch, m=m, n=n, k=k)
    _, i = oracle.gemm(a, b, sr, nthreads=0)
    dc = synth.uniform_f32(700 + seed, (batch, m, n), -1.0, 1.0)
    return a, b, dc, i


@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 5, 7, 3), (3, 70, 45, 37), (1, 40, 33, 300),
                                   (2, 129, 65, 130), (1, 8, 300, 700)])
def test_backward_matches_oracle(trop, sr, shape):
    a, b, dc, i = _case(sr, *shape)
    da, db = trop.gemm_backward(_dev(a), _dev(b), _dev(dc), _dev(i), sr)
    ra, rb = oracle.gemm_backward(a, b, dc, i, sr)
    assert da.cpu().numpy().tobytes() == ra.tobytes()
    assert db.cpu().numpy().tobytes() == rb.tobytes()


@pytest.mark.parametrize("sr", SR)
def test_backward_full_size_batched_workload(trop, sr):
    """batch 64 x 256^3 (the benchmarked GEMM), the argmax from the GPU forward."""
    a, b = synth.gemm_batched_inputs(sr)
    ad, bd = _dev(a), _dev(b)
    _, i = trop.gemm(ad, bd, sr)
    dc = synth.uniform_f32(711, i.shape, -1.0, 1.0)
    da, db = trop.gemm_backward(ad, bd, _dev(dc), i, sr)
    ra, rb = oracle.gemm_backward(a, b, dc, i.cpu().numpy(), sr)
    assert da.cpu().numpy().tobytes() == ra.tobytes()
    assert db.cpu().numpy().tobytes() == rb.tobytes()
    # each gradient alone (max-times dB alone takes the lane walk with gathered factors)
    da1, db1 = trop.gemm_backward(ad, bd, _dev(dc), i, sr, want_b=False)
    assert db1 is None and da1.cpu().numpy().tobytes() == ra.tobytes()
    da1, db1 = trop.gemm_backward(ad, bd, _dev(dc), i, sr, want_a=False)
    assert da1 is None and db1.cpu().numpy().tobytes() == rb.tobytes()


def test_backward_strided_operands_and_outputs(trop):
    a, b, dc, i = _case(2, 2, 48, 40, 150, seed=3)
    # dC / argmax as transposed views of [b, n, m] storage, A as a transposed view too
    dct = _dev(np.ascontiguousarray(dc.transpose(0, 2, 1))).transpose(1, 2)
    it = _dev(np.ascontiguousarray(i.transpose(0, 2, 1))).transpose(1, 2)
    at = _dev(np.ascontiguousarray(a.transpose(0, 2, 1))).transpose(1, 2)
    oa = torch.empty((2, 150, 48), device="cuda").transpose(1, 2)     # dA written through strides
    ob = torch.empty((2, 40, 150), device="cuda").transpose(1, 2)     # dB likewise
    da, db = trop.gemm_backward(at, _dev(b), dct, it, 2, out_a=oa, out_b=ob)
    ra, rb = oracle.gemm_backward(a, b, dc, i, 2)
    np.testing.assert_array_equal(da.cpu().numpy(), ra)
    np.testing.assert_array_equal(db.cpu().numpy(), rb)


@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 5, 7, 3), (3, 70, 45, 37), (1, 40, 33, 300), (2, 129, 65, 130)])
def test_backward_one_gradient_matches_oracle(trop, sr, shape):
    """dA alone and dB alone, every semiring; K = 300 takes two bin spans."""
    a, b, dc, i = _case(sr, *shape, seed=9)
    ra, rb = oracle.gemm_backward(a, b, dc, i, sr)
    da, db = trop.gemm_backward(_dev(a), _dev(b), _dev(dc), _dev(i), sr, want_b=False)
    assert db is None and da.cpu().numpy().tobytes() == ra.tobytes()
    da, db = trop.gemm_backward(_dev(a), _dev(b), _dev(dc), _dev(i), sr, want_a=False)
    assert da is None and db.cpu().numpy().tobytes() == rb.tobytes()


def test_backward_maxtimes_gradient_of_b_alone_strided_with_out_of_range_indices(trop):
    """max-times dB alone through transposed views of A, dC, the argmax and dB, with indices that
    route nowhere (-1, K) and K = 300 (two bin spans): the factor gathers follow A's strides."""
    a, b, dc, i = _case(2, 2, 48, 40, 300, seed=4)
    i = i.copy()
    i[0, 3, :5] = -1
    i[1, 4, 5:9] = 300
    dct = _dev(np.ascontiguousarray(dc.transpose(0, 2, 1))).transpose(1, 2)
    it = _dev(np.ascontiguousarray(i.transpose(0, 2, 1))).transpose(1, 2)
    at = _dev(np.ascontiguousarray(a.transpose(0, 2, 1))).transpose(1, 2)
    ob = torch.empty((2, 40, 300), device="cuda").transpose(1, 2)
    da, db = trop.gemm_backward(at, _dev(b), dct, it, 2, want_a=False, out_b=ob)
    _, rb = oracle.gemm_backward(a, b, dc, i, 2)
    assert da is None
    assert db.cpu().numpy().tobytes() == rb.tobytes()


def test_backward_one_side_and_out_of_range_indices(trop):
    a, b, dc, i = _case(0, 1, 20, 30, 10, seed=5)
    i = i.copy()
    i[0, 3, :5] = -1          # routes nowhere
    i[0, 4, 5:9] = 10         # == K: routes nowhere
    da, db = trop.gemm_backward(_dev(a), _dev(b), _dev(dc), _dev(i), 0, want_b=False)
    ra, rb = oracle.gemm_backward(a, b, dc, i, 0)
    assert db is None
    np.testing.assert_array_equal(da.cpu().numpy(), ra)
    da, db = trop.gemm_backward(_dev(a), _dev(b), _dev(dc), _dev(i), 0, want_a=False)
    assert da is None
    np.testing.assert_array_equal(db.cpu().numpy(), rb)


def test_backward_empty_extents_zero_the_gradient(trop):
    # N = 0: nothing routes, dA must come back all zero
    da, db = trop.gemm_backward(torch.ones((2, 3, 4), device="cuda"), torch.ones((2, 4, 0), device="cuda"),
                                torch.empty((2, 3, 0), device="cuda"),
                                torch.empty((2, 3, 0), dtype=torch.int32, device="cuda"), 0)
    assert da.shape == (2, 3, 4) and (da.cpu().numpy() == 0).all()
    assert db.shape == (2, 4, 0)


@pytest.mark.parametrize("sr", SR)
def test_autograd_function_routes_through_the_argmax(trop, sr):
    a, b, dc, _ = _case(sr, 2, 30, 20, 50, seed=9)
    ta = _dev(a).requires_grad_(True)
    tb = _dev(b).requires_grad_(True)
    c = trop.TropicalGemm.apply(ta, tb, sr)
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    np.testing.assert_array_equal(c.detach().cpu().numpy(), rc)
    c.backward(_dev(dc))
    ra, rb = oracle.gemm_backward(a, b, dc, ri, sr)
    assert ta.grad.cpu().numpy().tobytes() == ra.tobytes()
    assert tb.grad.cpu().numpy().tobytes() == rb.tobytes()

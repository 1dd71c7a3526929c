"""Pins of the oracle's tropical GEMM backward (winner routing) to things other
than itself: hand-computed 2x2 gradients, the adjoint identity of the routing
(the rustytorch commit tests <S x, y> == <x, S^T y>), mass conservation, and
CPU autograd of the plain max/min definition on tie-free inputs."""

import numpy as np
import pytest
import torch

import oracle
import synth

A22 = np.array([[[1, 2], [3, 4]]], dtype=np.float32)
B22 = np.array([[[5, 6], [7, 8]]], dtype=np.float32)
ONES = np.ones((1, 2, 2), dtype=np.float32)


@pytest.mark.parametrize("sr,da,db", [
    # max-plus: every argmax is 1 -> all of dC goes to column 1 of A and row 1 of B
    (0, [[0, 2], [0, 2]], [[0, 0], [2, 2]]),
    # min-plus: every argmax is 0
    (1, [[2, 0], [2, 0]], [[2, 2], [0, 0]]),
    # max-times: argmax 1; dA[m,1] = sum_n B[1,n] = 7 + 8, dB[1,n] = sum_m A[m,1] = 2 + 4
    (2, [[0, 15], [0, 15]], [[0, 0], [6, 6]]),
])
def test_backward_hand_2x2(sr, da, db):
    _, i = oracle.gemm(A22, B22, sr)
    ga, gb = oracle.gemm_backward(A22, B22, ONES, i, sr)
    np.testing.assert_array_equal(ga[0], np.array(da, np.float32))
    np.testing.assert_array_equal(gb[0], np.array(db, np.float32))


@pytest.mark.parametrize("sr", [0, 1])
def test_backward_adjoint_identity_and_mass(sr):
    a, b = synth.gemm_batched_inputs(sr, batch=3, m=17, n=23, k=11)
    _, i = oracle.gemm(a, b, sr)
    dc = synth.uniform_int(901, i.shape, -5, 5).astype(np.float32)
    ga, gb = oracle.gemm_backward(a, b, dc, i, sr)
    x = synth.uniform_int(902, a.shape, -7, 7).astype(np.float64)
    y = synth.uniform_int(903, b.shape, -7, 7).astype(np.float64)
    bb, mm, nn = np.meshgrid(np.arange(3), np.arange(17), np.arange(23), indexing="ij")
    # <dA, X> = sum dC[b,m,n] X[b,m,I[b,m,n]]  and  <dB, Y> = sum dC[b,m,n] Y[b,I[b,m,n],n]
    assert (ga.astype(np.float64) * x).sum() == (dc * x[bb, mm, i]).sum()
    assert (gb.astype(np.float64) * y).sum() == (dc * y[bb, i, nn]).sum()
    # every output's gradient lands somewhere exactly once
    np.testing.assert_array_equal(ga.sum(axis=2), dc.sum(axis=2))
    np.testing.assert_array_equal(gb.sum(axis=1), dc.sum(axis=1))


@pytest.mark.parametrize("sr", [0, 1, 2])
def test_backward_matches_autograd_of_the_definition(sr):
    rng = np.random.default_rng(7 + sr)
    nb, m, k, n = 2, 9, 13, 7
    a = rng.uniform(0.5 if sr == 2 else -1, 1, (nb, m, k)).astype(np.float32)
    if sr == 2:
        b = (2.0 ** rng.integers(-3, 3, (nb, k, n))).astype(np.float32)   # exact products with integer dC
    else:
        b = rng.uniform(-1, 1, (nb, k, n)).astype(np.float32)
    dc = rng.integers(-4, 5, (nb, m, n)).astype(np.float32)
    ta = torch.tensor(a, requires_grad=True)
    tb = torch.tensor(b, requires_grad=True)
    t = ta[:, :, :, None] * tb[:, None, :, :] if sr == 2 else ta[:, :, :, None] + tb[:, None, :, :]
    c, idx = t.min(dim=2) if sr == 1 else t.max(dim=2)
    # tie-free inputs: the routing index of autograd is the unique optimum
    ref_c, ref_i = oracle.gemm(a, b, sr)
    np.testing.assert_array_equal(c.detach().numpy(), ref_c)
    np.testing.assert_array_equal(idx.numpy(), ref_i)
    c.backward(torch.tensor(dc))
    ga, gb = oracle.gemm_backward(a, b, dc, ref_i, sr)
    np.testing.assert_array_equal(ga, ta.grad.numpy())
    if sr == 2:
        # dB sums dC * A over m: products of arbitrary floats, whose f32 sum depends on the order
        # autograd happens to use; at most a few ulp apart
        np.testing.assert_allclose(gb, tb.grad.numpy(), rtol=4e-7 * m, atol=1e-6)
    else:
        np.testing.assert_array_equal(gb, tb.grad.numpy())


def test_backward_ignores_out_of_range_indices():
    a = np.zeros((1, 1, 3), np.float32)
    b = np.zeros((1, 3, 2), np.float32)
    i = np.array([[[5, -1]]], np.int32)
    ga, gb = oracle.gemm_backward(a, b, np.ones((1, 1, 2), np.float32), i, 0)
    assert not ga.any() and not gb.any()

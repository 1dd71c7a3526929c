"""GPU parity: permute / diagonal gather / trace reduce (tropical_permute_trace,
tropical_permute_pair) vs the CPU oracle, bit-exact, for f32 / i32 / i64."""

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

NP = {"f32": np.float32, "i32": np.int32, "i64": np.int64}


@pytest.fixture(scope="module")
def trop():
    import einsum_device_side_gb300 as t
    t.load()
    return t


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _perm_spec(perm):
    src = "abcdefghijklmnop"[:len(perm)]
    return src + "->" + "".join(src[p] for p in perm)


@pytest.mark.parametrize("dtype", ["f32", "i32", "i64"])
@pytest.mark.parametrize("dims,perm", [
    ((16,) * 6, None),                         # the benchmarked rank-6 shape, seeded permutation
    ((3, 70, 65), (2, 0, 1)),                  # ragged transpose tiles
    ((5, 4, 3, 2, 7), (4, 3, 2, 1, 0)),
    ((64, 64), (1, 0)),
    ((33, 1, 17, 9), (1, 3, 0, 2)),            # unit axis
    ((8, 9, 10), (0, 2, 1)),
    ((6, 7, 128), (1, 0, 2)),                  # innermost axis kept: row copy
    ((2, 3, 5, 7, 11, 13), (5, 1, 3, 0, 2, 4)),
])
def test_permute_matches_oracle(trop, dtype, dims, perm):
    x, p = synth.permute_inputs(dtype, dims=dims)
    perm = list(p if perm is None else perm)
    spec = _perm_spec(perm)
    y = trop.permute_trace(_dev(x), spec)
    ref, _ = oracle.einsum(spec, x, nthreads=0)
    assert y.cpu().numpy().tobytes() == ref.tobytes()
    # permute o inverse permute = identity, bitwise, on the device
    inv = list(np.argsort(perm))
    src = spec.split("->")[1]
    back = trop.permute_trace(y, src + "->" + "".join(src[i] for i in inv))
    assert back.cpu().numpy().tobytes() == x.tobytes()


def test_permute_strided_input_and_output(trop):
    x, _ = synth.permute_inputs("f32", dims=(10, 12, 14))
    xd = _dev(x)[:, ::2, 1:]                       # non-contiguous view
    out = torch.empty((10, 6, 13), device="cuda").permute(0, 2, 1)   # (10, 13, 6), strided
    y = trop.permute_trace(xd, "abc->acb", out=out)
    ref, _ = oracle.einsum("abc->acb", x[:, ::2, 1:], nthreads=0)     # the oracle walks the strided view
    assert y.cpu().numpy().tobytes() == ref.tobytes()


@pytest.mark.parametrize("sr", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["f32", "i32", "i64"])
@pytest.mark.parametrize("spec", ["iijk->ijk", "iijk->jk", "iijk->kj", "iijk->", "ijkl->li", "iij->i", "aab->ba"])
def test_trace_matches_oracle(trop, sr, dtype, spec):
    shapes = {"iijk->ijk": (12, 12, 9, 10), "iijk->jk": (12, 12, 9, 10), "iijk->kj": (12, 12, 9, 10),
              "iijk->": (12, 12, 9, 10), "ijkl->li": (5, 300, 7, 9), "iij->i": (40, 40, 3000),
              "aab->ba": (7, 7, 5)}
    shp = shapes[spec]
    if dtype == "f32":
        x = synth.uniform_f32(31, shp, 0.0 if sr == 2 else -1.0, 1.0)
    else:
        x = synth.uniform_int(32, shp, 0 if sr == 2 else -1000, 1000, NP[dtype])
    y, a = trop.permute_trace(_dev(x), spec, sr, argmax=True)
    ref, refa = oracle.einsum(spec, x, semiring=sr, nthreads=0)
    assert y.cpu().numpy().tobytes() == ref.tobytes()
    np.testing.assert_array_equal(a.cpu().numpy(), refa)


def test_trace_workload_full_size(trop):
    x = synth.trace_inputs()
    xd = _dev(x)
    y = trop.permute_trace(xd, "iijk->ijk")
    ref, _ = oracle.einsum("iijk->ijk", x, nthreads=0)
    assert y.cpu().numpy().tobytes() == ref.tobytes()
    y2, a2 = trop.permute_trace(xd, "iijk->jk", "maxplus", argmax=True)
    ref2, refa2 = oracle.einsum("iijk->jk", x, nthreads=0)
    np.testing.assert_array_equal(y2.cpu().numpy(), ref2)
    np.testing.assert_array_equal(a2.cpu().numpy(), refa2)


@pytest.mark.parametrize("sr", [0, 1])
def test_full_reduction_with_argmax_large(trop, sr):
    x = synth.uniform_f32(77, (1 << 22,), -1, 1)
    x[3_000_000] = 5.0
    x[3_500_000] = 5.0                                  # tie: first one wins
    x[3_100_000] = -5.0
    x[3_600_000] = -5.0
    x2 = x.reshape(1024, 4096)
    y, a = trop.permute_trace(_dev(x2), "ij->", sr, argmax=True)
    ref, refa = oracle.einsum("ij->", x2, semiring=sr, nthreads=0)
    assert y.cpu().numpy().tobytes() == ref.tobytes()
    assert int(a.item()) == int(refa) == (3_000_000 if sr == 0 else 3_100_000)


def test_empty_reduction_and_empty_output(trop):
    x = torch.empty((0, 5), device="cuda")
    y, a = trop.permute_trace(x, "ij->j", "maxplus", argmax=True)
    assert (y.cpu().numpy() == -np.inf).all() and (a.cpu().numpy() == 0).all()
    y = trop.permute_trace(torch.empty((5, 0), device="cuda"), "ij->ji")
    assert y.shape == (0, 5)


def test_permute_pair_one_mapping(trop):
    v = synth.uniform_f32(5, (9, 70, 33), -1, 1)
    g = synth.uniform_int(6, (9, 70, 33), 0, 1 << 30, np.int32)
    rv, _ = oracle.einsum("abc->cab", v, nthreads=0)
    rg, _ = oracle.einsum("abc->cab", g, nthreads=0)
    ov, og = trop.permute_pair(_dev(v), _dev(g), "abc->cab")
    assert ov.cpu().numpy().tobytes() == rv.tobytes()
    np.testing.assert_array_equal(og.cpu().numpy(), rg)
    # companion with its own strides (a transposed view) still follows the same index map
    gd = _dev(np.ascontiguousarray(np.transpose(g, (1, 0, 2)))).permute(1, 0, 2)
    ov, og = trop.permute_pair(_dev(v), gd, "abc->cab")
    np.testing.assert_array_equal(og.cpu().numpy(), rg)


@pytest.mark.parametrize("sr", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["f32", "i32", "i64"])
@pytest.mark.parametrize("spec,shape", [("ijk->k", (300, 5, 70)), ("ij->j", (100, 33)), ("iijk->jk", (128, 128, 3, 40))])
def test_reduce_over_slices_with_ties(trop, sr, dtype, spec, shape):
    """Reductions whose outputs are contiguous in the input run as coalesced
    slices merged in shared memory; small integer ranges force ties, so the
    merge must keep the first index."""
    lo = 0 if sr == 2 else -3
    if dtype == "f32":
        x = synth.uniform_int(41, shape, lo, 3).astype(np.float32)
    else:
        x = synth.uniform_int(42, shape, lo, 3, NP[dtype])
    y, a = trop.permute_trace(_dev(x), spec, sr, argmax=True)
    ref, refa = oracle.einsum(spec, x, semiring=sr, nthreads=0)
    assert y.cpu().numpy().tobytes() == ref.tobytes()
    np.testing.assert_array_equal(a.cpu().numpy(), refa)

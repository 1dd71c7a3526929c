"""The allocation-free trace entry point (tropical_permute_trace_noalloc).

It serves callers of this library that cannot let it allocate device memory
(hosts that own every device allocation, loops that cannot absorb an
allocation's implicit synchronisation, processes whose device memory is
already handed to their own allocator).  The test calls it through the C ABI
on two calls in a row -- the fixed scratch it shares between calls keeps the
previous call's contents -- and checks each result against the CPU oracle and
against what tropical_permute_trace returns.  Kept in a file that pytest
collects last.
"""

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

SR = {"maxplus": 0, "minplus": 1, "maxtimes": 2}


@pytest.fixture(scope="module")
def trop():
    import einsum_device_side_gb300 as t
    t.load()
    return t


# 'ij->' (one output) and 'iij->i' (a diagonal whose output stride in the input is not 1)
# split each output's reduced range into partials that live in the fixed scratch; the two
# tile-path cases ('ijk->k', 'iijk->jk', outputs contiguous in the input) never touch it.
CASES = [
    ("ij->", (1024, 4096), "maxplus", "f32"),
    ("iij->i", (40, 40, 3000), "minplus", "f32"),
    ("ij->", (512, 4096), "minplus", "i32"),
    ("iij->i", (40, 40, 3000), "maxplus", "i32"),
    ("ij->", (512, 4096), "maxplus", "i64"),
    ("iij->i", (40, 40, 3000), "minplus", "i64"),
    ("ij->", (512, 4096), "maxtimes", "f64"),
    ("iij->i", (40, 40, 3000), "maxplus", "f64"),
    ("ijk->k", (64, 300, 16), "maxplus", "i64"),
    ("iijk->jk", (128, 128, 8, 8), "maxplus", "i32"),
]


def _input(shape, dtype, seed, sr):
    lo = 0 if sr == "maxtimes" else -1
    if dtype == "f32":
        return synth.uniform_f32(seed, shape, float(lo), 1.0)
    if dtype == "f64":
        return synth.uniform_f64(seed, shape, float(lo), 1.0)
    np_dt = np.int32 if dtype == "i32" else np.int64
    return synth.uniform_int(seed, shape, lo * 1000, 1000, np_dt)


@pytest.mark.parametrize("spec,shape,sr,dtype", CASES)
def test_noalloc_matches_oracle_and_pooled_entry_point_twice(trop, spec, shape, sr, dtype):
    for call, seed in enumerate((901, 902)):           # two calls in a row, different data
        x_np = _input(shape, dtype, seed + len(shape), sr)
        x = torch.from_numpy(x_np).cuda()
        ref, ref_arg = trop.permute_trace(x, spec, sr, argmax=True)
        out = torch.empty_like(ref)
        arg = torch.empty_like(ref_arg)
        trop.permute_trace_noalloc(x, spec, sr, out=out, argmax=arg)
        torch.cuda.synchronize()
        want, want_arg = oracle.einsum(spec, x_np, semiring=SR[sr], nthreads=0)
        assert out.cpu().numpy().tobytes() == want.tobytes(), f"values differ from the oracle on call {call}"
        np.testing.assert_array_equal(arg.cpu().numpy(), want_arg, err_msg=f"argmax vs oracle, call {call}")
        assert torch.equal(out, ref), f"values differ from tropical_permute_trace on call {call}"
        assert torch.equal(arg, ref_arg), f"argmax differs from tropical_permute_trace on call {call}"


@pytest.mark.parametrize("dtype", ["f32", "i64"])
def test_noalloc_without_argmax(trop, dtype):
    x_np = _input((40, 40, 3000), dtype, 77, "maxplus")
    x = torch.from_numpy(x_np).cuda()
    out = torch.empty((40,), dtype=x.dtype, device="cuda")
    for _ in range(2):
        got = trop.permute_trace_noalloc(x, "iij->i", "maxplus", out=out)
        torch.cuda.synchronize()
        want, _ = oracle.einsum("iij->i", x_np, semiring=0, nthreads=0)
        assert got.cpu().numpy().tobytes() == want.tobytes()


def test_noalloc_does_not_touch_the_pool(trop):
    x_np = _input((1024, 4096), "f32", 7, "maxplus")
    x = torch.from_numpy(x_np).cuda()
    out = torch.empty((), device="cuda")
    arg = torch.empty((), dtype=torch.int32, device="cuda")
    trop.permute_trace_noalloc(x, "ij->", "maxplus", out=out, argmax=arg)   # first call: address set-up
    torch.cuda.synchronize()
    before = trop.stats()["pool_allocs"]
    trop.permute_trace_noalloc(x, "ij->", "maxplus", out=out, argmax=arg)
    torch.cuda.synchronize()
    assert trop.stats()["pool_allocs"] == before
    want, want_arg = oracle.einsum("ij->", x_np, semiring=0, nthreads=0)
    assert out.cpu().numpy().tobytes() == want.tobytes()
    assert int(arg.item()) == int(want_arg)

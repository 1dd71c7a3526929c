"""The allocation-free trace entry point (tropical_permute_trace_noalloc).

It serves callers of this library that cannot let it allocate device memory.
The test calls it through the C ABI and checks that it returns exactly what
tropical_permute_trace returns, on two calls in a row (the fixed scratch it
shares between calls keeps the previous call's contents).  Kept in a file
that pytest collects last.
"""

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def trop():
    import einsum_device_side_gb300 as t
    t.load()
    return t


CASES = [
    ("ij->", (1024, 4096), "maxplus", "f32"),      # one output, 4M reduced: split into many partials
    ("iij->i", (40, 40, 3000), "minplus", "f32"),  # few outputs, long reduction
    ("ijk->k", (64, 300, 16), "maxplus", "i64"),
    ("iijk->jk", (128, 128, 8, 8), "maxplus", "i32"),
]


def _input(shape, dtype, seed):
    if dtype == "f32":
        return torch.from_numpy(synth.uniform_f32(seed, shape, -1.0, 1.0)).cuda()
    np_dt = np.int32 if dtype == "i32" else np.int64
    return torch.from_numpy(synth.uniform_int(seed, shape, -1000, 1000, np_dt)).cuda()


@pytest.mark.parametrize("spec,shape,sr,dtype", CASES)
def test_noalloc_matches_pooled_entry_point_twice(trop, spec, shape, sr, dtype):
    for call, seed in enumerate((901, 902)):           # two calls in a row, different data
        x = _input(shape, dtype, seed + len(shape))
        ref, ref_arg = trop.permute_trace(x, spec, sr, argmax=True)
        out = torch.empty_like(ref)
        arg = torch.empty_like(ref_arg)
        trop.permute_trace_noalloc(x, spec, sr, out=out, argmax=arg)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"values differ on call {call}"
        assert torch.equal(arg, ref_arg), f"argmax differs on call {call}"


def test_noalloc_does_not_touch_the_pool(trop):
    x = _input((1024, 4096), "f32", 7)
    out = torch.empty((), device="cuda")
    arg = torch.empty((), dtype=torch.int32, device="cuda")
    trop.permute_trace_noalloc(x, "ij->", "maxplus", out=out, argmax=arg)   # first call: address set-up
    torch.cuda.synchronize()
    before = trop.stats()["pool_allocs"]
    trop.permute_trace_noalloc(x, "ij->", "maxplus", out=out, argmax=arg)
    torch.cuda.synchronize()
    assert trop.stats()["pool_allocs"] == before
    assert float(out.item()) == float(x.max().item())
    assert int(arg.item()) == int(torch.argmax(x.reshape(-1)).item())

"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module only draws numbers: it holds none of the tropical arithmetic, so
both sides can take their inputs from it without sharing any method code.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014).  Output i of the stream with seed s is the
SplitMix64 mix of ``s + (i + 1) * 0x9E3779B97F4A7C15`` (mod 2**64), so any
prefix can be drawn in one vectorised numpy pass.

Recipes (one stream per tensor, ``seed = 0x7E570000 + 16 * workload + tensor``):

* f32 uniform(a, b): ``a + (b - a) * (z >> 40) * 2**-24``.  For (a, b) = (-1, 1)
  and (0, 1) every value is exactly representable in binary32, and (-1, 1)
  never yields -0.0.
* f64 uniform(a, b): ``a + (b - a) * (z >> 11) * 2**-53``.  For (-1, 1) and
  (0, 1) every value is exactly representable in binary64 (and uses the whole
  53-bit significand, so binary32 arithmetic would round differently); (-1, 1)
  never yields -0.0.
* integers uniform in [lo, hi]: ``lo + z % n`` with rejection of the top
  partial block (``z >= 2**64 - 2**64 % n``), consuming the stream in order.
* axis permutations: Fisher-Yates, swapping position i with ``z % (i + 1)``
  for i = n-1 .. 1 (the tiny modulo bias is irrelevant for test inputs).
* spin-glass couplings: one coupling per draw, ``+1`` if the top bit is set
  else ``-1``; horizontal bonds row-major, then vertical bonds row-major.
"""

from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

BASE_SEED = 0x7E570000

# Workload numbers used to derive seeds (one per benchmark workload).
W_GEMM64 = 0        # single 64^3 max-plus GEMM with argmax + transpose
W_GEMM_BATCHED = 1  # batch 64 x 256^3, three semirings
W_PERMUTE = 2       # rank-6 16^6 permute and (128,128,64,64) trace
W_EINSUM = 3        # 'zacd,zdce->zea'
W_ISING = 4         # 24x24 spin glass


def seed_for(workload: int, tensor: int) -> int:
    return BASE_SEED + 16 * workload + tensor


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset .. offset+n-1 of the SplitMix64 stream with this seed."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform_f32(seed: int, shape, lo: float, hi: float) -> np.ndarray:
    n = int(np.prod(shape, dtype=np.int64))
    z = splitmix64(seed, n)
    u = (z >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
    x = lo + (hi - lo) * u
    return x.astype(np.float32).reshape(shape)


def uniform_f64(seed: int, shape, lo: float, hi: float) -> np.ndarray:
    n = int(np.prod(shape, dtype=np.int64))
    z = splitmix64(seed, n)
    u = (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return (lo + (hi - lo) * u).reshape(shape)


def uniform_int(seed: int, shape, lo: int, hi: int, dtype=np.int32) -> np.ndarray:
    n = int(np.prod(shape, dtype=np.int64))
    span = hi - lo + 1
    assert span >= 1
    limit = (1 << 64) - ((1 << 64) % span)
    out = np.empty(0, dtype=np.uint64)
    offset = 0
    while out.size < n:
        need = n - out.size
        z = splitmix64(seed, need + 64, offset)
        offset += need + 64
        if limit < (1 << 64):
            z = z[z < np.uint64(limit)]
        out = np.concatenate([out, z])
    vals = (out[:n] % np.uint64(span)).astype(np.int64) + lo
    return vals.astype(dtype).reshape(shape)


def permutation(seed: int, n: int, reject_identity: bool = True) -> list:
    offset = 0
    while True:
        z = splitmix64(seed, n, offset)
        offset += n
        p = list(range(n))
        for i in range(n - 1, 0, -1):
            j = int(z[n - 1 - i] % np.uint64(i + 1))
            p[i], p[j] = p[j], p[i]
        if not reject_identity or p != list(range(n)) or n <= 1:
            return p


def couplings(seed: int, rows: int, cols: int):
    """(Jh, Jv): Jh[r][c] couples (r,c)-(r,c+1), Jv[r][c] couples (r,c)-(r+1,c)."""
    nh = rows * (cols - 1)
    nv = (rows - 1) * cols
    z = splitmix64(seed, nh + nv)
    bits = (z >> np.uint64(63)).astype(np.int8)
    j = (2 * bits - 1).astype(np.int8)
    jh = j[:nh].reshape(rows, cols - 1).copy()
    jv = j[nh:].reshape(rows - 1, cols).copy()
    return jh, jv


# ---------------------------------------------------------------------------
# The benchmark workloads (sizes and value distributions only).

def gemm64_inputs():
    """64x64x64, integers in [-8, 8] stored as f32 (forces argmax ties)."""
    s = W_GEMM64
    a = uniform_int(seed_for(s, 0), (1, 64, 64), -8, 8).astype(np.float32)
    b = uniform_int(seed_for(s, 1), (1, 64, 64), -8, 8).astype(np.float32)
    return a, b


SEMIRING_RANGES = {0: (-1.0, 1.0), 1: (-1.0, 1.0), 2: (0.0, 1.0)}


def gemm_batched_inputs(semiring: int, batch=64, m=256, n=256, k=256, dtype="f32"):
    lo, hi = SEMIRING_RANGES[semiring]
    s = W_GEMM_BATCHED
    draw = uniform_f64 if dtype == "f64" else uniform_f32
    a = draw(seed_for(s, 2 * semiring), (batch, m, k), lo, hi)
    b = draw(seed_for(s, 2 * semiring + 1), (batch, k, n), lo, hi)
    return a, b


def permute_inputs(dtype: str, dims=(16,) * 6):
    s = W_PERMUTE
    if dtype == "f32":
        x = uniform_f32(seed_for(s, 0), dims, -1.0, 1.0)
    elif dtype == "i32":
        x = uniform_int(seed_for(s, 1), dims, -1000, 1000, np.int32)
    elif dtype == "i64":
        x = uniform_int(seed_for(s, 2), dims, -1000, 1000, np.int64)
    else:
        raise ValueError(dtype)
    perm = permutation(seed_for(s, 3), len(dims))
    return x, perm


def trace_inputs(shape=(128, 128, 64, 64)):
    return uniform_f32(seed_for(W_PERMUTE, 4), shape, -1.0, 1.0)


def einsum_inputs(z=16, a=512, e=512, c=32, d=32):
    s = W_EINSUM
    A = uniform_f32(seed_for(s, 0), (z, a, c, d), -1.0, 1.0)
    B = uniform_f32(seed_for(s, 1), (z, d, c, e), -1.0, 1.0)
    return A, B


def ising_couplings(rows=24, cols=24):
    return couplings(seed_for(W_ISING, 0), rows, cols)

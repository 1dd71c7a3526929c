"""CPU oracle for the tropical einsum hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
library under test never imports it, and it imports nothing from the
library: the two share no code (inputs come from ``synth``).

The arithmetic lives in ``oracle.c`` (plain C, one binary32 rounding per
tropical product, strict-compare running result); this file only builds that
library with gcc and marshals numpy arrays into it.  See ``oracle.c`` for the
definitions and the passages of the pages each one follows.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MAXPLUS, MINPLUS, MAXTIMES = 0, 1, 2
SEMIRINGS = {"maxplus": MAXPLUS, "minplus": MINPLUS, "maxtimes": MAXTIMES}

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP if available)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    try:
        subprocess.run(base + ["-fopenmp", src, "-o", tmp, "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64p = ctypes.POINTER(ctypes.c_int64)
            i32p = ctypes.POINTER(ctypes.c_int32)
            lib.oracle_einsum.restype = ctypes.c_int
            lib.oracle_einsum.argtypes = [
                ctypes.c_int, ctypes.c_int,
                ctypes.c_int, i32p, i64p, i64p, P,
                ctypes.c_int, i32p, i64p, i64p, P,
                ctypes.c_int, i32p, P, i32p,
                i64p, ctypes.c_int64, ctypes.c_int]
            i8p = ctypes.POINTER(ctypes.c_int8)
            lib.oracle_ising_energy.restype = ctypes.c_int64
            lib.oracle_ising_energy.argtypes = [ctypes.c_int, ctypes.c_int, i8p, i8p, i8p]
            lib.oracle_ising_brute.restype = ctypes.c_int
            lib.oracle_ising_brute.argtypes = [ctypes.c_int, ctypes.c_int, i8p, i8p, i64p, i8p]
            lib.oracle_ising_ground.restype = ctypes.c_int
            lib.oracle_ising_ground.argtypes = [ctypes.c_int, ctypes.c_int, i8p, i8p, i64p, i8p,
                                                ctypes.c_int]
            I64 = ctypes.c_int64
            lib.oracle_gemm_backward.restype = ctypes.c_int
            lib.oracle_gemm_backward.argtypes = [ctypes.c_int, I64, I64, I64, I64] + [P, I64, I64, I64] * 6
            _lib = lib
    return _lib


def _arr(ctype, values):
    values = list(values)
    return (ctype * max(1, len(values)))(*values)


_DTYPES = {np.dtype(np.float32): 0, np.dtype(np.int32): 1, np.dtype(np.int64): 2, np.dtype(np.float64): 3}


def parse_spec(spec: str):
    """'ab,bc->ac' -> ([labels...], ...), labels as ints (code points)."""
    if "->" not in spec:
        raise ValueError("spec needs an explicit '->'")
    lhs, rhs = spec.replace(" ", "").split("->")
    ops = lhs.split(",")
    return [[ord(ch) for ch in op] for op in ops], [ord(ch) for ch in rhs]


def einsum(spec, a: np.ndarray, b: np.ndarray | None = None, semiring: int = MAXPLUS,
           samples=None, nthreads: int = 1, out_labels=None):
    """Tropical einsum by direct definition.  ``spec`` is either an einsum string
    or a tuple (labels_a, labels_b_or_None, labels_out) of int label lists.

    Returns (values, argmax).  Without ``samples`` both have the output's shape
    (row-major in the output label order); with ``samples`` (output linear
    indices) both are 1-D, one entry per sample."""
    lib = _load()
    if isinstance(spec, str):
        ops, lo = parse_spec(spec)
        la = ops[0]
        lb = ops[1] if len(ops) > 1 else None
    else:
        la, lb, lo = spec
    if (lb is None) != (b is None):
        raise ValueError("operand count does not match the spec")
    if len(la) != a.ndim or (b is not None and len(lb) != b.ndim):
        raise ValueError("rank does not match the spec")
    dt = _DTYPES[a.dtype]
    if b is not None and b.dtype != a.dtype:
        raise ValueError("dtype mismatch")
    sizes = {}
    for l, s in zip(la, a.shape):
        sizes.setdefault(l, s)
    if b is not None:
        for l, s in zip(lb, b.shape):
            sizes.setdefault(l, s)
    out_shape = tuple(int(sizes[l]) for l in lo)
    isz = a.itemsize
    st_a = [s // isz for s in a.strides]
    if samples is None:
        out = np.empty(out_shape, dtype=a.dtype)
        arg = np.empty(out_shape, dtype=np.int32)
        samp_ptr, ns = None, 0
    else:
        samples = np.ascontiguousarray(samples, dtype=np.int64)
        out = np.empty(samples.shape[0], dtype=a.dtype)
        arg = np.empty(samples.shape[0], dtype=np.int32)
        samp_ptr = samples.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        ns = samples.shape[0]
    if b is not None:
        st_b = [s // isz for s in b.strides]
        nb, lbp, shb, stb, bp = (len(lb), _arr(ctypes.c_int32, lb), _arr(ctypes.c_int64, b.shape),
                                 _arr(ctypes.c_int64, st_b), b.ctypes.data)
    else:
        nb, lbp, shb, stb, bp = -1, None, None, None, None
    rc = lib.oracle_einsum(int(semiring), dt,
                           len(la), _arr(ctypes.c_int32, la), _arr(ctypes.c_int64, a.shape),
                           _arr(ctypes.c_int64, st_a), a.ctypes.data,
                           nb, lbp, shb, stb, bp,
                           len(lo), _arr(ctypes.c_int32, lo), out.ctypes.data,
                           arg.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                           samp_ptr, ns, int(nthreads))
    if rc == -5:
        raise OverflowError("an integer tropical product falls outside the operand type "
                            "(the inputs violate the no-overflow precondition)")
    if rc != 0:
        raise ValueError(f"oracle_einsum failed with code {rc}")
    return out, arg


def gemm(a: np.ndarray, b: np.ndarray, semiring: int = MAXPLUS, samples=None, nthreads: int = 1):
    """Batched tropical GEMM C[b,m,n] = (+)_k A[b,m,k] (x) B[b,k,n] with argmax k
    (the einsum 'bmk,bkn->bmn'); accepts strided numpy views."""
    return einsum("bmk,bkn->bmn", a, b, semiring, samples=samples, nthreads=nthreads)


def gemm_backward(a: np.ndarray, b: np.ndarray, dc: np.ndarray, argmax: np.ndarray, semiring: int = MAXPLUS,
                  want_a: bool = True, want_b: bool = True):
    """Gradient of C[b,m,n] = (+)_k A[b,m,k] (x) B[b,k,n] with respect to A and B,
    routed through the forward argmax (see oracle.c, oracle_gemm_backward).
    Returns (dA, dB); either is None when not wanted."""
    lib = _load()
    a = np.asarray(a, dtype=np.float32)
    b = np.asarray(b, dtype=np.float32)
    dc = np.asarray(dc, dtype=np.float32)
    argmax = np.asarray(argmax, dtype=np.int32)
    nb, m, k = a.shape
    n = b.shape[2]
    assert b.shape == (nb, k, n) and dc.shape == (nb, m, n) and argmax.shape == (nb, m, n)
    da = np.empty((nb, m, k), dtype=np.float32) if want_a else None
    db = np.empty((nb, k, n), dtype=np.float32) if want_b else None

    def ptr_st(x):
        if x is None:
            return [None, 0, 0, 0]
        s = [st // x.itemsize for st in x.strides]
        return [x.ctypes.data, s[0], s[1], s[2]]
    rc = lib.oracle_gemm_backward(int(semiring), nb, m, n, k, *ptr_st(a), *ptr_st(b), *ptr_st(dc),
                                  *ptr_st(argmax), *ptr_st(da), *ptr_st(db))
    assert rc == 0
    return da, db


def _i8(x):
    x = np.ascontiguousarray(x, dtype=np.int8)
    return x, x.ctypes.data_as(ctypes.POINTER(ctypes.c_int8))


def ising_energy(jh, jv, spins) -> int:
    """H(s) = -sum J s_i s_j over the open-boundary grid (spins +-1, shape (R, C))."""
    lib = _load()
    spins = np.asarray(spins)
    r, c = spins.shape
    jh, pjh = _i8(jh)
    jv, pjv = _i8(jv)
    s, ps = _i8(spins)
    return int(lib.oracle_ising_energy(r, c, pjh, pjv, ps))


def ising_brute(jh, jv, rows: int, cols: int):
    """(W, spins): W = max over all configurations of sum J s_i s_j (exhaustive)."""
    lib = _load()
    jh, pjh = _i8(jh)
    jv, pjv = _i8(jv)
    spins = np.zeros((rows, cols), dtype=np.int8)
    w = ctypes.c_int64(0)
    rc = lib.oracle_ising_brute(rows, cols, pjh, pjv, ctypes.byref(w),
                                spins.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)))
    if rc != 0:
        raise ValueError(f"oracle_ising_brute failed with code {rc}")
    return int(w.value), spins


def ising_ground(jh, jv, rows: int, cols: int, nthreads: int = 0):
    """(W, spins) by site-by-site max-plus elimination with back-tracking."""
    lib = _load()
    jh, pjh = _i8(jh)
    jv, pjv = _i8(jv)
    spins = np.zeros((rows, cols), dtype=np.int8)
    w = ctypes.c_int64(0)
    rc = lib.oracle_ising_ground(rows, cols, pjh, pjv, ctypes.byref(w),
                                 spins.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_ising_ground failed with code {rc}")
    return int(w.value), spins

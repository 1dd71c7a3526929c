"""Device-resident tropical einsum for GB300 (sm_103a): thin Python binding.

Every function here marshals torch CUDA tensors into the C ABI declared in
``include/tropical.h`` and calls ``libtropical_gb300.so``; all computation
runs in that library's CUDA kernels.  There is no CPU fallback: if the
library is missing the first call raises.

Semirings: ``"maxplus"`` (max, +), ``"minplus"`` (min, +), ``"maxtimes"``
(max, *).  Argmax tensors are int32.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

__all__ = [
    "TropicalError", "load", "permute_trace", "permute_pair", "gemm", "einsum", "contract_tree",
    "tree_backtrack", "stats", "reset_stats", "sync_pool", "release_pool", "plan_describe", "version",
    "SEMIRINGS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtropical_gb300.so")
# the bounds-checked build (build.py --debug), loaded instead when TROP_LIBRARY=debug
LIB_DEBUG_PATH = os.path.join(_HERE, "_build_debug", "libtropical_gb300.so")
SEMIRINGS = {"maxplus": 0, "minplus": 1, "maxtimes": 2}
_DTYPES = {torch.float32: 0, torch.int32: 1, torch.int64: 2, torch.float64: 3}
MAX_RANK = 32

ERRORS = {
    -1: "INVALID_ARG", -2: "HOST_POINTER", -3: "DEVICE_MISMATCH", -4: "DTYPE", -5: "SHAPE", -6: "SPEC",
    -7: "OVERFLOW", -8: "CUDA", -9: "OOM", -10: "UNSUPPORTED",
}


class TropicalError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{ERRORS.get(code, code)}: {message}")
        self.code = code
        self.name = ERRORS.get(code, str(code))


class TropTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("shape", ctypes.c_int64 * MAX_RANK), ("stride", ctypes.c_int64 * MAX_RANK)]


class TropNode(ctypes.Structure):
    _fields_ = [("lhs", ctypes.c_int32), ("rhs", ctypes.c_int32), ("n_lhs", ctypes.c_int32),
                ("n_rhs", ctypes.c_int32), ("n_out", ctypes.c_int32),
                ("lhs_labels", ctypes.POINTER(ctypes.c_int32)), ("rhs_labels", ctypes.POINTER(ctypes.c_int32)),
                ("out_labels", ctypes.POINTER(ctypes.c_int32))]


_STAT_FIELDS = ["module_inits", "kernel_launches", "pool_allocs", "pool_hits", "pool_device_mallocs",
                "pool_retired", "pool_released", "pool_event_waits", "pool_leaked", "pool_bytes_cached",
                "stream_syncs", "plan_cache_hits", "plan_cache_misses", "gemm_early_starts"]


class TropStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in _STAT_FIELDS]


_lib = None
_fc = None  # the CPython binding of the hot entry points (csrc/fastcall.c), when built


def _load_fastcall(lib_path: str):
    """The fast-call extension built beside the library (None if this Python had no headers
    to build it with; the ctypes binding then serves every call)."""
    import glob
    import importlib.machinery
    import importlib.util
    found = glob.glob(os.path.join(os.path.dirname(lib_path), "_fastcall*.so"))
    if not found:
        return None
    loader = importlib.machinery.ExtensionFileLoader("_fastcall", found[0])
    spec = importlib.util.spec_from_file_location("_fastcall", found[0], loader=loader)
    mod = importlib.util.module_from_spec(spec)
    loader.exec_module(mod)
    return mod


def load(path: str | None = None):
    """Load the shared library (once).  Raises if it has not been built.  With TROP_LIBRARY=debug
    in the environment the bounds-checked build is loaded instead (through ctypes only)."""
    global _lib, _fc
    if _lib is not None:
        return _lib
    debug = os.environ.get("TROP_LIBRARY", "") == "debug"
    path = path or (LIB_DEBUG_PATH if debug else LIB_PATH)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m einsum_device_side_gb300.build` "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    TP = ctypes.POINTER(TropTensor)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64p = ctypes.POINTER(ctypes.c_int64)
    sig = {
        "tropical_init": (I, [I]),
        "tropical_permute_trace": (I, [TP, ctypes.c_char_p, I, TP, P, P]),
        "tropical_permute_pair": (I, [TP, TP, ctypes.c_char_p, TP, TP, P]),
        "tropical_permute_trace_noalloc": (I, [TP, ctypes.c_char_p, I, TP, P, P]),
        "tropical_gemm_strided_batched_argmax": (I, [I, I, I64, I64, I64, I64, P, I64, I64, I64, P, I64, I64, I64,
                                                     P, I64, I64, I64, P, P]),
        "tropical_einsum_pairwise": (I, [ctypes.c_char_p, TP, TP, I, TP, P, P]),
        "tropical_gemm_backward": (I, [I, I64, I64, I64, I64, P, I64, I64, I64, P, I64, I64, I64,
                                       P, I64, I64, I64, P, P, I64, I64, I64, P, I64, I64, I64, P]),
        "tropical_contract_tree": (I, [I, TP, I, ctypes.POINTER(TropNode), I, TP, ctypes.POINTER(P), P]),
        "tropical_tree_backtrack": (I, [I, TP, I, ctypes.POINTER(TropNode), ctypes.POINTER(P), I64, I, P, P]),
        "tropical_tree_plan_create": (I, [I, TP, I, ctypes.POINTER(TropNode), I, TP, ctypes.POINTER(P),
                                          ctypes.POINTER(P)]),
        "tropical_tree_plan_run": (I, [P, P]),
        "tropical_tree_plan_info": (I, [P, i64p, ctypes.POINTER(ctypes.c_size_t)]),
        "tropical_tree_plan_destroy": (I, [P]),
        "tropical_sync_pool": (I, []),
        "tropical_release_pool": (I, []),
        "tropical_stats": (I, [ctypes.POINTER(TropStats)]),
        "tropical_reset_stats": (None, []),
        "tropical_last_error": (ctypes.c_char_p, []),
        "tropical_version": (I, []),
        "tropical_plan_describe": (I, [ctypes.c_char_p, I, i64p, i64p, I, i64p, i64p, ctypes.c_char_p, I]),
        "tropical_debug_fail_next_event_records": (None, [I]),
        "tropical_set_pool_capacity": (None, [I]),
        "tropical_set_plan_cache_capacity": (None, [I]),
        "tropical_device_wait_timeouts": (I, [ctypes.POINTER(ctypes.c_uint), I]),
        "tropical_debug_set_wait_mode": (None, [I]),
        "tropical_debug_bounds_report": (I, [ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_int),
                                             ctypes.POINTER(ctypes.c_uint64), I]),
        "tropical_debug_bounds_trim": (I, [I64]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    del i32p
    _lib = lib
    _fc = None if debug else _load_fastcall(path)
    if _fc is not None:
        _fc.set_torch_handles(torch.float32, torch.int32, torch.int64, torch.float64,
                              _raw_stream or (lambda dev: torch.cuda.current_stream(dev).cuda_stream))
    return lib


def _check(rc: int):
    if rc != 0:
        msg = _lib.tropical_last_error().decode(errors="replace")
        raise TropicalError(rc, msg)


_SPECS: dict = {}


def _spec(spec: str) -> bytes:
    b = _SPECS.get(spec)
    if b is None:
        if len(_SPECS) >= 4096:
            _SPECS.clear()
        b = _SPECS[spec] = spec.encode()
    return b


def _dt(t: torch.Tensor) -> int:
    code = _DTYPES.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return code


def _ptr(t) -> int | None:
    return t.data_ptr() if t is not None and t.numel() else None


def _sr(semiring) -> int:
    if semiring.__class__ is str:
        return SEMIRINGS[semiring]
    return int(semiring)


# the current stream's raw handle without building a Stream object (a few us per call)
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None, like: torch.Tensor | None = None) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        dev = like.get_device() if like is not None else -1
        return _raw_stream(dev if dev >= 0 else torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


_desc_cache: dict = {}


def tensor_desc(t: torch.Tensor) -> TropTensor:
    """The C descriptor of a tensor.  A descriptor is a pure function of (data
    pointer, dtype, shape, strides), so repeated calls on the same tensors reuse
    one (bounded cache; the C side only reads it)."""
    key = (t.data_ptr(), t.dtype, t.shape, t.stride())
    d = _desc_cache.get(key)
    if d is None:
        if len(_desc_cache) >= 4096:
            _desc_cache.clear()
        d = _desc_cache[key] = _make_desc(t)
    return d


def _make_desc(t: torch.Tensor) -> TropTensor:
    code = _DTYPES.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    n = t.dim()
    if n > MAX_RANK:
        raise ValueError("rank above 32")
    d = TropTensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = code
    d.rank = n
    if n:
        d.shape[:n] = t.shape
        d.stride[:n] = t.stride()
    return d


def _spec_shape(spec: str, shapes):
    lhs, out = spec.replace(" ", "").split("->")
    sizes = {}
    for op, shp in zip(lhs.split(","), shapes):
        for ch, s in zip(op, shp):
            sizes.setdefault(ch, s)
    missing = [ch for ch in out if ch not in sizes]
    if missing:
        raise TropicalError(-6, f"output label(s) {''.join(missing)} appear in no operand of '{spec}'")
    return [sizes[ch] for ch in out]


def _check_argmax(am: torch.Tensor, out: torch.Tensor, like: torch.Tensor, contiguous: bool = True):
    """The C ABI writes an int32 argmax in out's shape (contiguous row-major, or
    with out's strides for the GEMM): anything else would be written past its end
    or read back wrongly, so it is refused here."""
    if am.dtype != torch.int32:
        raise TropicalError(-4, f"argmax must be int32, got {am.dtype}")
    if am.shape != out.shape:
        raise TropicalError(-5, f"argmax shape {tuple(am.shape)} differs from out shape {tuple(out.shape)}")
    if am.get_device() != like.get_device():
        raise TropicalError(-3, f"argmax is on {am.device}, operands on {like.device}")
    if contiguous and not am.is_contiguous():
        raise TropicalError(-1, "argmax must be contiguous (row-major in out's shape)")


def permute_trace(x: torch.Tensor, spec: str, semiring="maxplus", out: torch.Tensor | None = None,
                  argmax: bool | torch.Tensor = False, stream=None):
    """Unary permute / diagonal gather / tropical trace.  Returns ``out`` or
    ``(out, argmax)`` when ``argmax`` is True or a tensor."""
    lib = _lib or load()
    if out is None:
        out = torch.empty(_spec_shape(spec, [x.shape]), dtype=x.dtype, device=x.device)
    am = None
    if argmax is not False:
        if isinstance(argmax, torch.Tensor):
            am = argmax
            _check_argmax(am, out, x)
        elif argmax:
            am = torch.empty(out.shape, dtype=torch.int32, device=x.device)
    if _fc is not None:
        # the binding reads the tensors' data_ptr(), dtype, shape and stride() itself (data_ptr()
        # of an empty tensor may be 0: the C ABI accepts NULL data when an extent is 0)
        rc = _fc.permute_trace_t(x, spec, semiring, out, am, stream, False)
    else:
        dx, do = tensor_desc(x), tensor_desc(out)
        rc = lib.tropical_permute_trace(ctypes.byref(dx), _spec(spec), _sr(semiring), ctypes.byref(do), _ptr(am),
                                        _stream(stream, x))
    if rc:
        _check(rc)
    return (out, am) if am is not None else out


def permute_trace_noalloc(x: torch.Tensor, spec: str, semiring="maxplus", *, out: torch.Tensor,
                          argmax: torch.Tensor | None = None, stream=None):
    """Like permute_trace, but the library allocates nothing: for callers that
    cannot let it allocate device memory.  ``out`` (and ``argmax``, if wanted)
    must be given; split reductions use the library's fixed scratch, so calls
    must not overlap on the GPU."""
    lib = _lib or load()
    if argmax is not None:
        _check_argmax(argmax, out, x)
    if _fc is not None:
        rc = _fc.permute_trace_t(x, spec, semiring, out, argmax, stream, True)
    else:
        dx, do = tensor_desc(x), tensor_desc(out)
        rc = lib.tropical_permute_trace_noalloc(ctypes.byref(dx), _spec(spec), _sr(semiring), ctypes.byref(do),
                                                _ptr(argmax), _stream(stream, x))
    _check(rc)
    return (out, argmax) if argmax is not None else out


def permute_pair(val: torch.Tensor, arg: torch.Tensor, spec: str, out_val=None, out_arg=None, stream=None):
    """Permute a result and its int32 argmax through one index mapping."""
    lib = _lib or load()
    if out_val is None or out_arg is None:
        shape = _spec_shape(spec, [val.shape])
        if out_val is None:
            out_val = torch.empty(shape, dtype=val.dtype, device=val.device)
        if out_arg is None:
            out_arg = torch.empty(shape, dtype=torch.int32, device=val.device)
    if _fc is not None:
        rc = _fc.permute_pair_t(val, arg, spec, out_val, out_arg, stream)
    else:
        a, b, c, d = tensor_desc(val), tensor_desc(arg), tensor_desc(out_val), tensor_desc(out_arg)
        rc = lib.tropical_permute_pair(ctypes.byref(a), ctypes.byref(b), _spec(spec), ctypes.byref(c),
                                       ctypes.byref(d), _stream(stream, val))
    _check(rc)
    return out_val, out_arg


def gemm(A: torch.Tensor, B: torch.Tensor, semiring="maxplus", argmax: bool = True, out=None, out_argmax=None,
         stream=None):
    """Strided-batched tropical GEMM: A [batch, M, K], B [batch, K, N] (any
    strides, batch stride 0 allowed).  Returns (C, argmax) or C."""
    lib = _lib or load()
    if A.dim() == 2:
        A = A.unsqueeze(0)
    if B.dim() == 2:
        B = B.unsqueeze(0)
    batch = max(A.shape[0], B.shape[0])
    if A.shape[0] != batch:
        A = A.expand(batch, *A.shape[1:])
    if B.shape[0] != batch:
        B = B.expand(batch, *B.shape[1:])
    M, K = A.shape[1], A.shape[2]
    N = B.shape[2]
    if B.shape[1] != K:
        raise ValueError("inner extents differ")
    if A.dtype not in _DTYPES or B.dtype != A.dtype:
        raise TypeError(f"gemm needs two operands of one dtype (float32, float64, int32, int64), "
                        f"got {A.dtype} and {B.dtype}")
    if out is None:
        out = torch.empty((batch, M, N), dtype=A.dtype, device=A.device)
    elif out.dtype != A.dtype:
        raise TypeError(f"out is {out.dtype}, operands are {A.dtype}")
    am = None
    if argmax:
        am = out_argmax if out_argmax is not None else torch.empty((batch, M, N), dtype=torch.int32, device=A.device)
        _check_argmax(am, out, A, contiguous=False)
        if am.stride() != out.stride():
            raise ValueError("argmax must have the strides of out")
    sa, sb, so = A.stride(), B.stride(), out.stride()
    call = _fc.gemm if _fc is not None else lib.tropical_gemm_strided_batched_argmax
    dev = out.get_device()
    st = stream.cuda_stream if stream is not None else (_raw_stream(dev) if dev >= 0 and _raw_stream
                                                        else _stream(None, out))
    rc = call(SEMIRINGS.get(semiring, semiring), _DTYPES[A.dtype], batch, M, N, K, A.data_ptr(), sa[0], sa[1],
              sa[2], B.data_ptr(), sb[0], sb[1], sb[2], out.data_ptr(), so[0], so[1], so[2],
              None if am is None else am.data_ptr(), st)
    if rc:
        _check(rc)
    return (out, am) if argmax else out


def gemm_backward(A: torch.Tensor, B: torch.Tensor, dC: torch.Tensor, argmax: torch.Tensor, semiring="maxplus",
                  want_a: bool = True, want_b: bool = True, out_a=None, out_b=None, stream=None):
    """Gradient of the strided-batched tropical GEMM C = A (x) B with respect to A
    and B, routed through the forward argmax (dA: [batch, M, K], dB: [batch, K,
    N]).  Returns (dA, dB); an unwanted one is None."""
    lib = load()
    if A.dim() == 2:
        A = A.unsqueeze(0)
    if B.dim() == 2:
        B = B.unsqueeze(0)
    if dC.dim() == 2:
        dC, argmax = dC.unsqueeze(0), argmax.unsqueeze(0)
    batch, M, N = dC.shape
    K = A.shape[2]
    if A.shape[0] != batch:
        A = A.expand(batch, *A.shape[1:])
    if B.shape[0] != batch:
        B = B.expand(batch, *B.shape[1:])
    if argmax.shape != dC.shape or argmax.stride() != dC.stride():
        raise ValueError("argmax must have the shape and strides of dC")
    da = (out_a if out_a is not None else torch.empty((batch, M, K), device=dC.device)) if want_a else None
    db = (out_b if out_b is not None else torch.empty((batch, K, N), device=dC.device)) if want_b else None
    ptr = lambda t: t.data_ptr() if t is not None and t.numel() else None  # noqa: E731
    st = lambda t: tuple(t.stride()) if t is not None else (0, 0, 0)  # noqa: E731
    _check(lib.tropical_gemm_backward(
        _sr(semiring), batch, M, N, K, ptr(A), *st(A), ptr(B), *st(B), ptr(dC), *st(dC), ptr(argmax),
        ptr(da), *st(da), ptr(db), *st(db), _stream(stream, dC)))
    return da, db


class TropicalGemm(torch.autograd.Function):
    """Autograd over the batched tropical GEMM: forward = gemm (value and argmax),
    backward = gemm_backward through the saved argmax (winner routing).
    ``TropicalGemm.apply(A, B, semiring)`` returns C; the argmax stays saved."""

    @staticmethod
    def forward(ctx, A, B, semiring="maxplus"):
        C, I = gemm(A, B, semiring)
        ctx.semiring = semiring
        ctx.save_for_backward(A, B, I)
        ctx.mark_non_differentiable(I)
        return C

    @staticmethod
    def backward(ctx, dC):
        A, B, I = ctx.saved_tensors
        dA, dB = gemm_backward(A, B, dC.contiguous(), I, ctx.semiring,
                               want_a=ctx.needs_input_grad[0], want_b=ctx.needs_input_grad[1])
        if dA is not None and A.dim() == 2:
            dA = dA[0]
        if dB is not None and B.dim() == 2:
            dB = dB[0]
        return dA, dB, None


def einsum(spec: str, A: torch.Tensor, B: torch.Tensor, semiring="maxplus", argmax: bool = True, out=None,
           out_argmax=None, stream=None):
    """Pairwise tropical einsum, e.g. ``einsum('zacd,zdce->zea', A, B)``.
    Returns (out, argmax) or out."""
    lib = _lib or load()
    if out is None:
        out = torch.empty(_spec_shape(spec, [A.shape, B.shape]), dtype=A.dtype, device=A.device)
    am = None
    if argmax:
        am = out_argmax if out_argmax is not None else torch.empty(out.shape, dtype=torch.int32, device=A.device)
        _check_argmax(am, out, A)
    st = _stream(stream, out)
    if _fc is not None:
        rc = _fc.einsum(_spec(spec), _ptr(A), _dt(A), A.shape, A.stride(), _ptr(B), _dt(B), B.shape, B.stride(),
                        _sr(semiring), _ptr(out), _dt(out), out.shape, out.stride(), _ptr(am), st)
    else:
        a, b, o = tensor_desc(A), tensor_desc(B), tensor_desc(out)
        rc = lib.tropical_einsum_pairwise(_spec(spec), ctypes.byref(a), ctypes.byref(b), _sr(semiring),
                                          ctypes.byref(o), _ptr(am), st)
    _check(rc)
    return (out, am) if argmax else out


_NODE_DTYPE = np.dtype({"names": ["lhs", "rhs", "n_lhs", "n_rhs", "n_out", "lhs_labels", "rhs_labels", "out_labels"],
                        "formats": ["<i4"] * 5 + ["<u8"] * 3,
                        "offsets": [TropNode.lhs.offset, TropNode.rhs.offset, TropNode.n_lhs.offset,
                                    TropNode.n_rhs.offset, TropNode.n_out.offset, TropNode.lhs_labels.offset,
                                    TropNode.rhs_labels.offset, TropNode.out_labels.offset],
                        "itemsize": ctypes.sizeof(TropNode)})


class _NodeTable:
    """The trop_node array of a node list, built in one pass: every label list
    lives in one int32 array and the nodes point into it.  Keeps both alive for
    one call."""

    def __init__(self, nodes):
        lh, rh, nl, nr, no, labs = [], [], [], [], [], []
        for lhs, rhs, ll, rl, ol in nodes:
            rl = rl or ()
            lh.append(lhs)
            rh.append(-1 if rhs is None else rhs)
            nl.append(len(ll))
            nr.append(len(rl))
            no.append(len(ol))
            labs.extend(ll)
            labs.extend(rl)
            labs.extend(ol)
        labs.append(0)  # every pointer, even of an empty list, stays inside the array
        self.labels = np.asarray(labs, dtype=np.int32)
        nl, nr, no = (np.asarray(v, dtype=np.int64) for v in (nl, nr, no))
        start = np.zeros(len(nodes), dtype=np.int64)
        np.cumsum((nl + nr + no)[:-1], out=start[1:])
        base = self.labels.ctypes.data
        t = np.zeros(len(nodes), dtype=_NODE_DTYPE)
        t["lhs"], t["rhs"], t["n_lhs"], t["n_rhs"], t["n_out"] = lh, rh, nl, nr, no
        t["lhs_labels"] = base + 4 * start
        t["rhs_labels"] = base + 4 * (start + nl)
        t["out_labels"] = base + 4 * (start + nl + nr)
        self.table = t
        self.arr = t.ctypes.data_as(ctypes.POINTER(TropNode))


def contract_tree(inputs, nodes, semiring="maxplus", out: torch.Tensor | None = None, node_argmax=None,
                  stream=None):
    """Run a contraction tree.  ``nodes``: list of (lhs_id, rhs_id_or_None,
    lhs_labels, rhs_labels_or_None, out_labels) with integer labels; ids
    0..len(inputs)-1 are inputs, len(inputs)+j is node j.  ``out`` must have
    the root node's shape.  ``node_argmax``: optional list of int32 tensors or
    None per node."""
    lib = load()
    descs = (TropTensor * max(1, len(inputs)))(*[tensor_desc(t) for t in inputs])
    table = _NodeTable(nodes)
    ams = None
    if node_argmax is not None:
        ams = (ctypes.c_void_p * len(nodes))(*[(t.data_ptr() if t is not None and t.numel() else None)
                                               for t in node_argmax])
    o = tensor_desc(out)
    _check(lib.tropical_contract_tree(len(inputs), descs, len(nodes), table.arr, _sr(semiring), ctypes.byref(o),
                                      ams, _stream(stream, out)))
    return out


class TreePlan:
    """A contraction tree lowered once and captured as one CUDA graph
    (tropical_tree_plan_*).  It binds the tensors given here: ``run()`` reads
    the inputs' current contents and writes ``out`` and the node argmax
    tensors, so refill inputs in place between runs.  The tensors are kept
    referenced for the plan's lifetime."""

    def __init__(self, inputs, nodes, semiring="maxplus", out: torch.Tensor | None = None, node_argmax=None):
        lib = load()
        self._keep = (list(inputs), out, None if node_argmax is None else list(node_argmax))
        descs = (TropTensor * max(1, len(inputs)))(*[tensor_desc(t) for t in inputs])
        table = _NodeTable(nodes)
        ams = None
        if node_argmax is not None:
            ams = (ctypes.c_void_p * len(nodes))(*[(t.data_ptr() if t is not None and t.numel() else None)
                                                   for t in node_argmax])
        o = tensor_desc(out)
        h = ctypes.c_void_p()
        _check(lib.tropical_tree_plan_create(len(inputs), descs, len(nodes), table.arr, _sr(semiring),
                                             ctypes.byref(o), ams, ctypes.byref(h)))
        self._h = h
        self.out = out
        k, w = ctypes.c_int64(), ctypes.c_size_t()
        _check(lib.tropical_tree_plan_info(h, ctypes.byref(k), ctypes.byref(w)))
        self.kernels, self.workspace_bytes = int(k.value), int(w.value)

    def run(self, stream=None):
        if self._h is None:
            raise RuntimeError("plan is closed")
        _check(_lib.tropical_tree_plan_run(self._h, _stream(stream, self.out)))
        return self.out

    def close(self):
        if getattr(self, "_h", None) is not None:
            _check(_lib.tropical_tree_plan_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tree_plan(inputs, nodes, semiring="maxplus", out: torch.Tensor | None = None, node_argmax=None) -> TreePlan:
    """Lower a contraction tree once and capture it as a CUDA graph; see TreePlan."""
    return TreePlan(inputs, nodes, semiring, out, node_argmax)


def tree_backtrack(inputs, nodes, node_argmax, n_labels: int, root_index: int = 0, assignment=None, stream=None):
    """Recover every eliminated label's value from the per-node argmaxes
    (device-side walk).  Returns an int32 device tensor of n_labels (-1 where
    undetermined)."""
    lib = load()
    dev = inputs[0].device if inputs else torch.device("cuda")
    if assignment is None:
        assignment = torch.empty(n_labels, dtype=torch.int32, device=dev)
    descs = (TropTensor * max(1, len(inputs)))(*[tensor_desc(t) for t in inputs])
    table = _NodeTable(nodes)
    ams = (ctypes.c_void_p * len(nodes))(*[(t.data_ptr() if t is not None and t.numel() else None)
                                           for t in node_argmax])
    _check(lib.tropical_tree_backtrack(len(inputs), descs, len(nodes), table.arr, ams, root_index, n_labels,
                                       assignment.data_ptr(), _stream(stream, assignment)))
    return assignment


def stats() -> dict:
    lib = load()
    s = TropStats()
    _check(lib.tropical_stats(ctypes.byref(s)))
    return {n: getattr(s, n) for n in _STAT_FIELDS}


def reset_stats():
    load().tropical_reset_stats()


def sync_pool():
    lib = load()
    _check(lib.tropical_sync_pool())


def release_pool():
    lib = load()
    _check(lib.tropical_release_pool())


def device_wait_timeouts(reset: bool = False) -> int:
    """Kernel waits on the current device that gave up since load (blocks until idle)."""
    n = ctypes.c_uint(0)
    _check(load().tropical_device_wait_timeouts(ctypes.byref(n), int(bool(reset))))
    return n.value


def set_plan_cache_capacity(n: int):
    """Bound of the pairwise einsum's plan cache (0 disables it)."""
    load().tropical_set_plan_cache_capacity(int(n))


def debug_set_wait_mode(mode: int):
    """Test hook: 1 = the TMA-fed GEMM's first operand wait gives up (then recovers), 2 = it
    then fails after its copies landed (the next call reports the error), 0 = normal."""
    load().tropical_debug_set_wait_mode(int(mode))


# translation units of the library, by the id the bounds-checked build records with a line
_BOUNDS_FILES = {1: "unary.cu", 2: "gemm.cu", 3: "gemm64.cu", 4: "gemm_int.cu", 5: "backward.cu", 6: "backtrack.cu"}


def debug_bounds_report(reset: bool = False) -> dict | None:
    """The bounds-checked build's violation record for the current device: {"count", "file",
    "line", "addr"} (the first violation's source location and address), or None from the
    normal build, which checks nothing.  Read once the work to inspect has completed."""
    lib = load()
    cnt, line, addr = ctypes.c_uint(0), ctypes.c_int(0), ctypes.c_uint64(0)
    rc = lib.tropical_debug_bounds_report(ctypes.byref(cnt), ctypes.byref(line), ctypes.byref(addr), int(reset))
    if rc == -10:  # TROP_ERR_UNSUPPORTED: the normal build
        return None
    _check(rc)
    return {"count": cnt.value, "file": _BOUNDS_FILES.get(line.value >> 16, "?"), "line": line.value & 0xFFFF,
            "addr": addr.value}


def debug_bounds_trim(nbytes: int) -> bool:
    """Test hook of the bounds-checked build: cut every byte range made from now on short by
    ``nbytes`` (0 restores exact ranges).  Returns False from the normal build."""
    rc = load().tropical_debug_bounds_trim(int(nbytes))
    if rc == -10:  # TROP_ERR_UNSUPPORTED: the normal build
        return False
    _check(rc)
    return True


def set_pool_capacity(n: int):
    load().tropical_set_pool_capacity(int(n))


def debug_fail_next_event_records(n: int):
    load().tropical_debug_fail_next_event_records(int(n))


def init(device: int = 0):
    lib = load()
    _check(lib.tropical_init(int(device)))


def version() -> int:
    return load().tropical_version()


def plan_describe(spec: str, shape_a, stride_a, shape_b, stride_b) -> str:
    """Host-only: how the pairwise einsum would be lowered (no GPU needed)."""
    lib = load()
    buf = ctypes.create_string_buffer(1024)
    arr = lambda v: (ctypes.c_int64 * max(1, len(v)))(*v)  # noqa: E731
    _check(lib.tropical_plan_describe(spec.encode(), len(shape_a), arr(shape_a), arr(stride_a), len(shape_b),
                                      arr(shape_b), arr(stride_b), buf, 1024))
    return buf.value.decode()

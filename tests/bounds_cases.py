"""Parity cases run against the bounds-checked build of the library.

Run as a script in a process of its own with TROP_LIBRARY=debug (the package then loads
``_build_debug/libtropical_gb300.so``): every stage of the path -- permutes (row copy,
tiled transpose, generic gather, value + argmax pairs), traces and reductions (per-thread,
tiled and split), the f32 GEMM on each of its routes (TMA-fed with the fused short-K resolve
or followed by the panel resolve, register-tiled with stream-K, streaming, generic), the f64 and integer GEMMs, the backward
in all three semirings, pairwise einsums and a contraction tree with back-tracking -- is
compared with the oracle, and the library's violation record is read at the end.  Prints
one JSON line: {"library", "cases", "failures": [...], "report": {...}}.
"""

from __future__ import annotations

import json
import os
import sys
import traceback

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main() -> int:
    import torch

    import einsum_device_side_gb300 as trop
    import oracle
    import synth
    from einsum_device_side_gb300 import ising

    lib_path = trop.LIB_DEBUG_PATH if os.environ.get("TROP_LIBRARY") == "debug" else trop.LIB_PATH
    trop.load()
    dev = torch.device("cuda:0")
    failures: list[str] = []
    ncases = 0

    def d(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    def same(name, got, want):
        if got.shape != want.shape or got.tobytes() != np.ascontiguousarray(want).tobytes():
            failures.append(name)

    def case(name, fn):
        nonlocal ncases
        ncases += 1
        try:
            fn()
        except Exception:  # a raised error is a failure of the case, not of the run
            failures.append(name + ": " + traceback.format_exc(limit=2).strip().splitlines()[-1])

    # ---- permutes: row copy, tiled transpose (f32, f64), generic gather, pairs
    def permute(dtype, dims, perm, strided=False):
        if dtype == "f64":
            x = synth.uniform_f64(synth.seed_for(synth.W_PERMUTE, 5), dims, -1.0, 1.0)
        else:
            x, _ = synth.permute_inputs(dtype, dims=dims)
        src = "abcdefgh"[:len(dims)]
        spec = src + "->" + "".join(src[p] for p in perm)
        xd = d(x)
        if strided:
            xd = d(np.concatenate([x, x], axis=-1))[..., ::2]
            x = np.ascontiguousarray(np.concatenate([x, x], axis=-1)[..., ::2])
        got = trop.permute_trace(xd, spec).cpu().numpy()
        same(f"permute {dtype} {dims} {perm}", got, np.transpose(x, perm))

    case("permute rows", lambda: permute("f32", (6, 5, 40), (1, 0, 2)))
    case("permute transpose f32", lambda: permute("f32", (33, 70, 9), (2, 1, 0)))
    case("permute transpose f64", lambda: permute("f64", (3, 65, 130), (0, 2, 1)))
    case("permute rank 6", lambda: permute("i32", (4, 5, 3, 6, 2, 4), (5, 2, 0, 4, 1, 3)))
    case("permute strided gather", lambda: permute("f32", (7, 9, 11), (2, 0, 1), strided=True))

    def pair():
        v = synth.uniform_f32(5, (9, 70, 33), -1, 1)
        g = synth.uniform_int(6, (9, 70, 33), 0, 1 << 30, np.int32)
        ov, og = trop.permute_pair(d(v), d(g), "abc->cab")
        same("pair values", ov.cpu().numpy(), np.transpose(v, (2, 0, 1)))
        same("pair argmax", og.cpu().numpy(), np.transpose(g, (2, 0, 1)))
    case("permute pair", pair)

    # ---- traces and reductions
    def reduce(spec, shape, sr, seed):
        x = synth.uniform_f32(seed, shape, 0.0 if sr == 2 else -1.0, 1.0)
        got, ga = trop.permute_trace(d(x), spec, sr, argmax=True)
        want, wa = oracle.einsum(spec, x, None, sr)
        same(f"reduce {spec} {shape} values", got.cpu().numpy(), want)
        same(f"reduce {spec} {shape} argmax", ga.cpu().numpy(), wa)

    for sr in (0, 1, 2):
        case(f"trace iijk->ijk sr{sr}", lambda sr=sr: reduce("iijk->ijk", (12, 12, 8, 16), sr, 31 + sr))
        case(f"reduce per thread sr{sr}", lambda sr=sr: reduce("ij->i", (5000, 20), sr, 34 + sr))
        case(f"reduce tiled sr{sr}", lambda sr=sr: reduce("ij->j", (700, 96), sr, 37 + sr))
        case(f"reduce split sr{sr}", lambda sr=sr: reduce("ij->i", (3, 300000), sr, 40 + sr))
        case(f"reduce full sr{sr}", lambda sr=sr: reduce("i->", (1 << 20,), sr, 43 + sr))

    # ---- GEMMs
    def gemm(sr, shape, dtype="f32", argmax=True, transpose_out=False):
        bt, m, n, k = shape
        a, b = synth.gemm_batched_inputs(sr, batch=bt, m=m, n=n, k=k, dtype=dtype)
        ad, bd = d(a), d(b)
        want, wa = oracle.gemm(a, b, sr, nthreads=0)
        if transpose_out:
            out = torch.empty((bt, n, m), dtype=ad.dtype, device=dev).transpose(1, 2)
            am = torch.empty((bt, n, m), dtype=torch.int32, device=dev).transpose(1, 2)
            c, i = trop.gemm(ad, bd, sr, out=out, out_argmax=am)
        elif argmax:
            c, i = trop.gemm(ad, bd, sr)
        else:
            c, i = trop.gemm(ad, bd, sr, argmax=False), None
        same(f"gemm {dtype} sr{sr} {shape} values", c.cpu().numpy(), want)
        if i is not None:
            same(f"gemm {dtype} sr{sr} {shape} argmax", i.cpu().numpy(), wa)

    for sr in (0, 1, 2):
        case(f"gemm TMA fused with the resolve sr{sr}", lambda sr=sr: gemm(sr, (64, 256, 256, 256)))
        case(f"gemm TMA + panel resolve sr{sr}", lambda sr=sr: gemm(sr, (32, 256, 256, 1024)))
        case(f"gemm tiled ragged sr{sr}", lambda sr=sr: gemm(sr, (3, 70, 45, 37)))
        case(f"gemm stream-K sr{sr}", lambda sr=sr: gemm(sr, (2, 129, 65, 1030)))
        case(f"gemm no argmax sr{sr}", lambda sr=sr: gemm(sr, (5, 200, 150, 90), argmax=False))
        case(f"gemm no argmax by TMA sr{sr}", lambda sr=sr: gemm(sr, (8, 128, 136, 64), argmax=False))
        case(f"gemm strided output sr{sr}", lambda sr=sr: gemm(sr, (2, 96, 80, 50), transpose_out=True))
        case(f"gemm thin M sr{sr}", lambda sr=sr: gemm(sr, (40, 3, 512, 64)))
        case(f"gemm f64 sr{sr}", lambda sr=sr: gemm(sr, (2, 70, 45, 37), dtype="f64"))

    def gemm_generic():
        a = synth.uniform_f32(50, (2, 9, 13), -1, 1)
        b = synth.uniform_f32(51, (2, 13, 11), -1, 1)
        ab = d(np.repeat(b, 2, axis=2))[:, :, ::2]  # column stride 2: the generic route
        c, i = trop.gemm(d(a), ab, 0)
        want, wa = oracle.gemm(a, b, 0, nthreads=0)
        same("gemm generic values", c.cpu().numpy(), want)
        same("gemm generic argmax", i.cpu().numpy(), wa)
    case("gemm generic strides", gemm_generic)

    def gemm_int(sr, dt, shape):
        bt, m, n, k = shape
        rng_hi = 1000
        lo = 0 if sr == 2 else -rng_hi
        a = synth.uniform_int(60 + sr, (bt, m, k), lo, rng_hi, dt)
        b = synth.uniform_int(63 + sr, (bt, k, n), lo, rng_hi, dt)
        c, i = trop.gemm(d(a), d(b), sr)
        want, wa = oracle.gemm(a, b, sr, nthreads=0)
        same(f"gemm {dt.__name__} sr{sr} values", c.cpu().numpy(), want)
        same(f"gemm {dt.__name__} sr{sr} argmax", i.cpu().numpy(), wa)

    for sr in (0, 1, 2):
        case(f"gemm i32 sr{sr}", lambda sr=sr: gemm_int(sr, np.int32, (3, 70, 45, 37)))
        case(f"gemm i64 sr{sr}", lambda sr=sr: gemm_int(sr, np.int64, (2, 33, 66, 130)))

    # ---- backward, every routing kernel
    def backward(sr, shape, seed):
        bt, m, n, k = shape
        a, b = synth.gemm_batched_inputs(sr, batch=bt, m=m, n=n, k=k)
        _, i = oracle.gemm(a, b, sr, nthreads=0)
        dc = synth.uniform_f32(700 + seed, (bt, m, n), -1.0, 1.0)
        da, db = trop.gemm_backward(d(a), d(b), d(dc), d(i), sr)
        ra, rb = oracle.gemm_backward(a, b, dc, i, sr)
        same(f"backward sr{sr} {shape} dA", da.cpu().numpy(), ra)
        same(f"backward sr{sr} {shape} dB", db.cpu().numpy(), rb)

    def backward_b_alone(sr, shape, seed):
        bt, m, n, k = shape
        a, b = synth.gemm_batched_inputs(sr, batch=bt, m=m, n=n, k=k)
        _, i = oracle.gemm(a, b, sr, nthreads=0)
        dc = synth.uniform_f32(700 + seed, (bt, m, n), -1.0, 1.0)
        _, db = trop.gemm_backward(d(a), d(b), d(dc), d(i), sr, want_a=False)
        _, rb = oracle.gemm_backward(a, b, dc, i, sr)
        same(f"backward dB alone sr{sr} {shape}", db.cpu().numpy(), rb)

    case("backward dB alone sr2", lambda: backward_b_alone(2, (3, 70, 45, 37), 11))
    case("backward dB alone long K sr2", lambda: backward_b_alone(2, (1, 40, 33, 300), 12))
    for sr in (0, 1, 2):
        case(f"backward sr{sr}", lambda sr=sr: backward(sr, (3, 70, 45, 37), sr))
        case(f"backward long K sr{sr}", lambda sr=sr: backward(sr, (1, 40, 33, 300), 3 + sr))
        case(f"backward wide sr{sr}", lambda sr=sr: backward(sr, (4, 64, 256, 128), 6 + sr))

    def backward_strided():
        a, b = synth.gemm_batched_inputs(2, batch=2, m=48, n=40, k=150)
        _, i = oracle.gemm(a, b, 2, nthreads=0)
        dc = synth.uniform_f32(709, (2, 48, 40), -1.0, 1.0)
        dct = d(np.ascontiguousarray(dc.transpose(0, 2, 1))).transpose(1, 2)
        it = d(np.ascontiguousarray(i.transpose(0, 2, 1))).transpose(1, 2)
        oa = torch.empty((2, 150, 48), device=dev).transpose(1, 2)
        ob = torch.empty((2, 40, 150), device=dev).transpose(1, 2)
        da, db = trop.gemm_backward(d(a), d(b), dct, it, 2, out_a=oa, out_b=ob)
        ra, rb = oracle.gemm_backward(a, b, dc, i, 2)
        same("backward strided dA", da.cpu().numpy(), ra)
        same("backward strided dB", db.cpu().numpy(), rb)
    case("backward strided", backward_strided)

    # ---- pairwise einsums
    def einsum(spec, sa, sb, sr, seed):
        lo = 0.0 if sr == 2 else -1.0
        a = synth.uniform_f32(seed, sa, lo, 1.0)
        b = synth.uniform_f32(seed + 1, sb, lo, 1.0)
        o, oa = trop.einsum(spec, d(a), d(b), sr)
        want, wa = oracle.einsum(spec, a, b, sr, nthreads=0)
        same(f"einsum {spec} values", o.cpu().numpy(), want)
        same(f"einsum {spec} argmax", oa.cpu().numpy(), wa)

    for sr in (0, 2):
        case(f"einsum zacd sr{sr}", lambda sr=sr: einsum("zacd,zdce->zea", (4, 40, 8, 8), (4, 8, 8, 30), sr, 80))
        case(f"einsum diagonal sr{sr}", lambda sr=sr: einsum("iij,jk->ki", (9, 9, 7), (7, 5), sr, 82))
        case(f"einsum reduce first sr{sr}", lambda sr=sr: einsum("ij,jk->k", (6, 8), (8, 5), sr, 84))
        case(f"einsum full sr{sr}", lambda sr=sr: einsum("abc,cab->", (3, 4, 5), (5, 3, 4), sr, 86))

    # ---- contraction tree with back-tracking
    def tree():
        jh, jv = synth.couplings(4, 8, 8)
        w, spins, _ = ising.ground_state(jh, jv)
        wo, so = oracle.ising_ground(jh, jv, 8, 8, nthreads=0)
        if w != wo or not np.array_equal(spins, so):
            failures.append("ising 8x8")
    case("contraction tree 8x8", tree)

    torch.cuda.synchronize()
    report = trop.debug_bounds_report()

    # the checks fire: with every range cut 4 bytes short, the last element of a permute's
    # input (or output) counts as outside -- its access is skipped and recorded
    control = None
    if trop.debug_bounds_trim(4):
        x = synth.uniform_f32(90, (8, 40, 6), -1.0, 1.0)
        trop.debug_bounds_report(reset=True)
        trop.permute_trace(d(x), "abc->cba")
        torch.cuda.synchronize()
        control = trop.debug_bounds_report(reset=True)
        trop.debug_bounds_trim(0)
    print(json.dumps({"library": lib_path, "cases": ncases, "failures": failures, "report": report,
                      "control": control}))
    return 0


if __name__ == "__main__":
    sys.exit(main())

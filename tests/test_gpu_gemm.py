"""GPU parity: strided-batched tropical GEMM with argmax vs the CPU oracle.

Values and argmax must be bit-identical (every tropical product rounds once,
max/min are exact, ties go to the smallest k).  Calls go through the C ABI
(tropical_gemm_strided_batched_argmax) via the ctypes binding.
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


def _check(trop, a, b, sr, a_dev=None, b_dev=None):
    a_dev = _dev(a) if a_dev is None else a_dev
    b_dev = _dev(b) if b_dev is None else b_dev
    c, i = trop.gemm(a_dev, b_dev, sr)
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    c, i = c.cpu().numpy(), i.cpu().numpy()
    assert c.tobytes() == rc.tobytes(), f"values differ at {np.argwhere(c != rc)[:5]}"
    np.testing.assert_array_equal(i, ri)


@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (1, 64, 64, 64), (3, 70, 45, 37), (2, 130, 129, 70),
                                   (1, 200, 65, 257), (4, 17, 300, 16), (2, 5, 7, 3), (1, 64, 64, 1),
                                   (2, 96, 80, 384), (1, 70, 130, 512), (1, 66, 40, 1032)])
def test_gemm_matches_oracle(trop, sr, shape):
    bt, m, n, k = shape
    a, b = synth.gemm_batched_inputs(sr, batch=bt, m=m, n=n, k=k)
    _check(trop, a, b, sr)


@pytest.mark.parametrize("sr", SR)
def test_gemm_integer_ties(trop, sr):
    # small integers force ties between different k: argmax must pick the first
    a = synth.uniform_int(11, (2, 96, 80), -3, 3).astype(np.float32)
    b = synth.uniform_int(12, (2, 80, 72), -3, 3).astype(np.float32)
    if sr == 2:
        a, b = np.abs(a), np.abs(b)
    _check(trop, a, b, sr)


def test_gemm64_workload_and_transpose_pair(trop):
    a, b = synth.gemm64_inputs()
    c, i = trop.gemm(_dev(a), _dev(b), 0)
    rc, ri = oracle.gemm(a, b, 0)
    np.testing.assert_array_equal(c.cpu().numpy(), rc)
    np.testing.assert_array_equal(i.cpu().numpy(), ri)
    ct, it = trop.permute_pair(c[0], i[0], "ij->ji")
    np.testing.assert_array_equal(ct.cpu().numpy(), rc[0].T)
    np.testing.assert_array_equal(it.cpu().numpy(), ri[0].T)


@pytest.mark.parametrize("layout", ["NT", "TN", "TT"])
def test_gemm_transposed_layouts(trop, layout):
    a, b = synth.gemm_batched_inputs(0, batch=2, m=96, n=80, k=50)
    ad, bd = _dev(a), _dev(b)
    if layout[0] == "T":
        ad = _dev(np.ascontiguousarray(np.swapaxes(a, 1, 2))).transpose(1, 2)
    if layout[1] == "T":
        bd = _dev(np.ascontiguousarray(np.swapaxes(b, 1, 2))).transpose(1, 2)
    _check(trop, a, b, 0, ad, bd)


def test_gemm_broadcast_batch_and_strided_output(trop):
    a, b = synth.gemm_batched_inputs(1, batch=3, m=40, n=33, k=21)
    b1 = b[:1]
    bd = _dev(b1).expand(3, 21, 33)
    out = torch.empty((3, 33, 40), dtype=torch.float32, device="cuda").transpose(1, 2)
    am = torch.empty((3, 33, 40), dtype=torch.int32, device="cuda").transpose(1, 2)
    c, i = trop.gemm(_dev(a), bd, 1, out=out, out_argmax=am)
    rc, ri = oracle.gemm(a, np.broadcast_to(b1, (3, 21, 33)), 1)
    np.testing.assert_array_equal(c.cpu().numpy(), rc)
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


@pytest.mark.parametrize("sr", SR)
def test_gemm_empty_contraction(trop, sr):
    a = torch.empty((2, 5, 0), device="cuda")
    b = torch.empty((2, 0, 7), device="cuda")
    c, i = trop.gemm(a, b, sr)
    zero = {0: -np.inf, 1: np.inf, 2: 0.0}[sr]
    assert (c.cpu().numpy() == np.float32(zero)).all() and (i.cpu().numpy() == 0).all()
    c, i = trop.gemm(torch.empty((2, 0, 3), device="cuda"), torch.empty((2, 3, 7), device="cuda"), sr)
    assert c.shape == (2, 0, 7)


def test_gemm_without_argmax_matches(trop):
    a, b = synth.gemm_batched_inputs(0, batch=2, m=70, n=90, k=45)
    c = trop.gemm(_dev(a), _dev(b), 0, argmax=False)
    rc, _ = oracle.gemm(a, b, 0)
    np.testing.assert_array_equal(c.cpu().numpy(), rc)


def test_identity_and_infinities(trop):
    rng = np.random.default_rng(3)
    a = rng.integers(-5, 6, size=(1, 70, 66)).astype(np.float32)
    eye = np.full((1, 66, 66), -np.inf, dtype=np.float32)
    eye[0, np.arange(66), np.arange(66)] = 0
    _check(trop, a, eye, 0)


@pytest.mark.parametrize("sr", SR)
def test_full_size_batched_workload(trop, sr):
    """batch 64 x 256^3 exactly as benchmarked: every output's value and argmax
    bitwise against the oracle (4,194,304 outputs per semiring), plus the argmax
    certificate A[m,I] (x) B[I,n] == C on the device."""
    a, b = synth.gemm_batched_inputs(sr)
    ad, bd = _dev(a), _dev(b)
    c, i = trop.gemm(ad, bd, sr)
    torch.cuda.synchronize()
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    assert c.cpu().numpy().tobytes() == rc.tobytes(), "values differ from the oracle"
    np.testing.assert_array_equal(i.cpu().numpy(), ri)
    idx = i.long()
    a_sel = torch.gather(ad, 2, idx)                                 # A[b, m, I[b,m,n]]
    b_sel = torch.gather(bd, 1, idx)                                 # B[b, I[b,m,n], n]
    t = a_sel * b_sel if sr == 2 else a_sel + b_sel
    assert torch.equal(t, c)


# ---------------------------------------------------------------- split tiles (stream-K) and the resolve pass

@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("batch,k,kernel", [(64, 256, "tma"), (128, 256, "tma"), (64, 248, "tiled"),
                                            (128, 248, "tiled")])
def test_plain_full_size(trop, sr, batch, k, kernel):
    """Batched 256 x 256 without argmax, every output vs the oracle.  K = 256: whole tiles by TMA
    (k_gemm_tma_plain).  K = 248 (not whole 16-wide k-tiles): the cp.async kernel, whose last
    partial wave is cut along k and the segments merged by the last CTA to finish."""
    a, b = synth.gemm_batched_inputs(sr, batch=batch, k=k)
    c = trop.gemm(_dev(a), _dev(b), sr, argmax=False)
    torch.cuda.synchronize()
    rc, _ = oracle.gemm(a, b, sr, nthreads=0)
    assert c.cpu().numpy().tobytes() == rc.tobytes()


@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("shape", [(1, 64, 64, 4096), (2, 100, 70, 2000), (1, 130, 64, 2001), (3, 64, 200, 520)])
def test_split_k_long_contraction(trop, sr, shape):
    """Few tiles and a long contraction: every tile is cut into many k segments
    (up to 32), and the argmax resolve walks several staged groups of B rows;
    K = 2001 is not a whole number of argmax chunks (generic resolve path)."""
    bt, m, n, k = shape
    a, b = synth.gemm_batched_inputs(sr, batch=bt, m=m, n=n, k=k)
    _check(trop, a, b, sr)
    c = trop.gemm(_dev(a), _dev(b), sr, argmax=False)
    rc, _ = oracle.gemm(a, b, sr, nthreads=0)
    assert c.cpu().numpy().tobytes() == rc.tobytes()


def test_split_k_strided_output(trop):
    """Output and argmax through transposed views (non-unit column strides): the
    merge stores and the generic resolve path."""
    a, b = synth.gemm_batched_inputs(0, batch=2, m=96, n=80, k=1536)
    ct = torch.empty((2, 80, 96), device="cuda")
    it = torch.empty((2, 80, 96), dtype=torch.int32, device="cuda")
    c, i = ct.transpose(1, 2), it.transpose(1, 2)
    trop.gemm(_dev(a), _dev(b), 0, out=c, out_argmax=i)
    rc, ri = oracle.gemm(a, b, 0, nthreads=0)
    np.testing.assert_array_equal(c.cpu().numpy(), rc)
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


def test_split_gemms_on_two_streams(trop):
    """Split GEMMs running at once on two streams use separate arrival counters:
    results equal the same calls made one after another."""
    work = []
    for s, (bt, m, n, k, arg) in enumerate([(64, 256, 256, 256, False), (1, 64, 128, 3072, True),
                                           (64, 256, 256, 256, False), (2, 64, 64, 2048, True)]):
        a, b = synth.gemm_batched_inputs(s % 3, batch=bt, m=m, n=n, k=k)
        work.append((s % 3, _dev(a), _dev(b), arg))
    ref = []
    for sr, ad, bd, arg in work:
        ref.append(trop.gemm(ad, bd, sr, argmax=arg))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for rep in range(3):
        for j, (sr, ad, bd, arg) in enumerate(work):
            with torch.cuda.stream(streams[j % 2]):
                outs.append((j, trop.gemm(ad, bd, sr, argmax=arg)))
    torch.cuda.synchronize()
    for j, got in outs:
        want = ref[j]
        if work[j][3]:
            assert torch.equal(got[0], want[0]) and torch.equal(got[1], want[1])
        else:
            assert torch.equal(got, want)


@pytest.mark.parametrize("sr", SR)
def test_whole_tiles_long_contraction(trop, sr):
    """Enough whole tiles that none is split, with K > 4096 (too many k-tiles to
    resolve the argmax inside the tile): chunk codes go through the separate
    resolve pass.  Every output's value and argmax vs the oracle."""
    a, b = synth.gemm_batched_inputs(sr, batch=60, m=128, n=128, k=4200)
    ad, bd = _dev(a), _dev(b)
    c, i = trop.gemm(ad, bd, sr)
    torch.cuda.synchronize()
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    assert c.cpu().numpy().tobytes() == rc.tobytes()
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


def test_argmax_gemm_streams_and_graph_replay(trop):
    """Whole-tile argmax GEMMs (value kernel + programmatic-dependent resolve
    pass): results must not depend on the stream a call runs on, on the order
    of problem sizes, or on replaying a captured CUDA graph with new inputs."""
    cases = [(0, 64, 256, 256, 256), (1, 8, 192, 320, 300), (2, 30, 128, 128, 512), (0, 40, 70, 200, 96)]
    work = []
    for sr, bt, m, n, k in cases:
        a, b = synth.gemm_batched_inputs(sr, batch=bt, m=m, n=n, k=k)
        work.append((sr, _dev(a), _dev(b)))
    ref = [trop.gemm(ad, bd, sr) for sr, ad, bd in work]
    torch.cuda.synchronize()
    for j, (sr, ad, bd) in enumerate(work[1:2] + work[3:4]):   # oracle pins for two of them
        got = ref[1] if j == 0 else ref[3]
        rc, ri = oracle.gemm(ad.cpu().numpy(), bd.cpu().numpy(), sr, nthreads=0)
        np.testing.assert_array_equal(got[0].cpu().numpy(), rc)
        np.testing.assert_array_equal(got[1].cpu().numpy(), ri)
    # fresh streams, problem sizes interleaved
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    order = [3, 1, 2, 0, 0, 2, 1, 3]
    outs = []
    for rep in range(2):
        for q, j in enumerate(order):
            sr, ad, bd = work[j]
            with torch.cuda.stream(streams[(q + rep) % 2]):
                outs.append((j, trop.gemm(ad, bd, sr)))
    torch.cuda.synchronize()
    for j, got in outs:
        assert torch.equal(got[0], ref[j][0]) and torch.equal(got[1], ref[j][1])
    # graph replay with new inputs copied in between replays
    sr, ad, bd = work[0]
    a2, b2 = synth.gemm_batched_inputs(1, batch=64, m=256, n=256, k=256)
    sets = [(ad, bd), (_dev(a2), _dev(b2))]
    ref2 = trop.gemm(sets[1][0], sets[1][1], sr)
    xa, xb = ad.clone(), bd.clone()
    c = torch.empty_like(ref[0][0])
    i = torch.empty_like(ref[0][1])
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        trop.gemm(xa, xb, sr, out=c, out_argmax=i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        trop.gemm(xa, xb, sr, out=c, out_argmax=i)
    for rep in range(4):
        src = sets[rep % 2]
        want = ref[0] if rep % 2 == 0 else ref2
        xa.copy_(src[0])
        xb.copy_(src[1])
        c.fill_(0)
        i.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(c, want[0]) and torch.equal(i, want[1]), rep


# ---------------------------------------------------------------- short contractions (K <= 256, whole chunks)
# These take the resolve pass that reads whole rows of A, one chunk per lane.

@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("shape", [(3, 70, 45, 40), (2, 130, 129, 248), (1, 33, 200, 256), (5, 64, 64, 8),
                                   (2, 191, 67, 136)])
def test_short_contraction_ragged(trop, sr, shape):
    bt, m, n, k = shape
    a, b = synth.gemm_batched_inputs(sr, batch=bt, m=m, n=n, k=k)
    _check(trop, a, b, sr)


@pytest.mark.parametrize("sr", SR)
def test_short_contraction_padded_rows_and_ties(trop, sr):
    """Integer entries (ties in every chunk), A and C/I rows padded past their extents,
    B broadcast over the batch: values and argmax against the oracle on the logical views."""
    bt, m, n, k = 3, 97, 75, 256
    a = synth.uniform_int(21, (bt, m, k), -4, 4).astype(np.float32)
    b = synth.uniform_int(22, (1, k, n), -4, 4).astype(np.float32)
    if sr == 2:
        a, b = np.abs(a), np.abs(b)
    wide = torch.zeros((bt, m, k + 12), dtype=torch.float32, device="cuda")
    wide[:, :, 4:4 + k] = _dev(a)
    ad = wide[:, :, 4:4 + k]                       # row stride k + 12, 16-byte aligned rows
    bd = _dev(b).expand(bt, k, n)
    cw = torch.empty((bt, m, n + 9), dtype=torch.float32, device="cuda")
    iw = torch.empty((bt, m, n + 9), dtype=torch.int32, device="cuda")
    c, i = trop.gemm(ad, bd, sr, out=cw[:, :, :n], out_argmax=iw[:, :, :n])
    rc, ri = oracle.gemm(a, np.broadcast_to(b, (bt, k, n)), sr, nthreads=0)
    assert c.cpu().numpy().tobytes() == np.ascontiguousarray(rc).tobytes()
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


@pytest.mark.parametrize("sr", SR)
def test_tma_gemm_given_up_wait_recovers_exactly(trop, sr):
    """A first operand wait that gives up is counted and waited again with the full bound:
    the results stay bit-exact against the oracle (test mode 1 makes every CTA's first wait
    give up at once)."""
    a, b = synth.gemm_batched_inputs(sr, batch=32)
    ad, bd = _dev(a), _dev(b)
    desc = trop.plan_describe("zmk,zkn->zmn", list(ad.shape), list(ad.stride()), list(bd.shape), list(bd.stride()))
    assert "kernel=tma" in desc, desc
    trop.device_wait_timeouts(reset=True)
    trop.debug_set_wait_mode(1)
    try:
        c, i = trop.gemm(ad, bd, sr)
        torch.cuda.synchronize()
    finally:
        trop.debug_set_wait_mode(0)
    assert trop.device_wait_timeouts(reset=True) == 32 * 4 * 4    # one per CTA (32 x 4 x 4 tiles)
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    assert c.cpu().numpy().tobytes() == rc.tobytes()
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


def test_tma_gemm_failed_wait_is_reported(trop):
    """When a wait cannot be completed the tile is abandoned and the failure reported by
    the next call (test mode 2 fails every CTA after its copies have landed, so nothing is
    in flight); the report comes once, and the next call is bit-exact again."""
    from einsum_device_side_gb300 import TropicalError
    a, b = synth.gemm_batched_inputs(0, batch=32)
    ad, bd = _dev(a), _dev(b)
    desc = trop.plan_describe("zmk,zkn->zmn", list(ad.shape), list(ad.stride()), list(bd.shape), list(bd.stride()))
    assert "kernel=tma" in desc, desc
    c = torch.full((32, 256, 256), 7.0, device="cuda")
    i = torch.full((32, 256, 256), -5, dtype=torch.int32, device="cuda")
    trop.debug_set_wait_mode(2)
    try:
        trop.gemm(ad, bd, 0, out=c, out_argmax=i)
        torch.cuda.synchronize()
    finally:
        trop.debug_set_wait_mode(0)
    assert bool((c == 7.0).all()), "an abandoned tile stores no values"
    assert bool((i == 0).all()), "an abandoned tile leaves no chunk code for the resolve pass"
    with pytest.raises(TropicalError) as ex:
        trop.gemm(ad, bd, 0, out=c, out_argmax=i)
    assert ex.value.name == "CUDA" and "abandoned" in str(ex.value)
    trop.device_wait_timeouts(reset=True)
    c2, i2 = trop.gemm(ad, bd, 0)                    # reported once: this call runs normally
    rc, ri = oracle.gemm(a, b, 0, nthreads=0)
    assert c2.cpu().numpy().tobytes() == rc.tobytes()
    np.testing.assert_array_equal(i2.cpu().numpy(), ri)


def test_tma_gemm_waits_never_gave_up(trop):
    """Every operand copy of the TMA-fed GEMM landed within its bounded wait (the device
    counter of given-up waits stays 0 after the full-size calls)."""
    for sr in SR:
        a, b = synth.gemm_batched_inputs(sr, batch=32)
        ad, bd = _dev(a), _dev(b)
        desc = trop.plan_describe("zmk,zkn->zmn", list(ad.shape), list(ad.stride()), list(bd.shape), list(bd.stride()))
        assert "kernel=tma" in desc, desc
        trop.gemm(ad, bd, sr)
    assert trop.device_wait_timeouts() == 0


# ---------------------------------------------------------------- the TMA-fed kernel (one batch axis, K % 16 == 0)

@pytest.mark.parametrize("sr", SR)
@pytest.mark.parametrize("shape", [(120, 70, 44, 48), (30, 130, 132, 256), (40, 200, 68, 128), (240, 64, 64, 16),
                                   (48, 33, 260, 512), (120, 65, 64, 1024)])
def test_tma_path_integer_ties_padded_rows(trop, sr, shape):
    """Small integers (ties between k in every chunk and across k-tiles), A's and the output's
    rows padded past their extents, ragged M and N: values and argmax equal the oracle's.  The
    batches give more than half a wave of tiles, so no tile is split along k and the planner
    confirms the layout takes the TMA-fed kernel (K = 512 and 1024 then take the panel
    resolve, the others the row resolve)."""
    bt, m, n, k = shape
    a = synth.uniform_int(41, (bt, m, k), -4, 4).astype(np.float32)
    b = synth.uniform_int(42, (bt, k, n), -4, 4).astype(np.float32)
    if sr == 2:
        a, b = np.abs(a), np.abs(b)
    wide = torch.zeros((bt, m, k + 8), dtype=torch.float32, device="cuda")
    wide[:, :, :k] = _dev(a)
    ad = wide[:, :, :k]                                   # row stride k + 8 (16-byte rows)
    bd = _dev(b)
    desc = trop.plan_describe("zmk,zkn->zmn", list(ad.shape), list(ad.stride()), list(bd.shape), list(bd.stride()))
    assert "kernel=tma" in desc, desc
    cw = torch.empty((bt, m, n + 4), dtype=torch.float32, device="cuda")
    iw = torch.empty((bt, m, n + 4), dtype=torch.int32, device="cuda")
    c, i = trop.gemm(ad, bd, sr, out=cw[:, :, :n], out_argmax=iw[:, :, :n])
    rc, ri = oracle.gemm(a, b, sr, nthreads=0)
    assert c.cpu().numpy().tobytes() == np.ascontiguousarray(rc).tobytes()
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


# ---------------------------------------------------------------- back-to-back one-launch GEMMs

def _gemm_set(sr, batch=24):
    """batch x 256^3: enough tiles for the TMA-fed kernel with its resolve in the same launch."""
    return synth.gemm_batched_inputs(sr, batch=batch)


def test_back_to_back_gemms_start_early_and_stay_exact(trop):
    """Three argmax GEMMs on one stream with disjoint buffers: the second and third read nothing
    the one before writes, so each starts loading and computing before that one has finished
    (gemm_early_starts), and every output still equals the oracle's, over repeated rounds."""
    sets = [_gemm_set(sr) for sr in SR]
    dev = [(_dev(a), _dev(b)) for a, b in sets]
    ref = [oracle.gemm(a, b, sr, nthreads=0) for sr, (a, b) in zip(SR, sets)]
    outs = [(torch.empty((24, 256, 256), device="cuda"), torch.empty((24, 256, 256), dtype=torch.int32, device="cuda"))
            for _ in SR]
    desc = trop.plan_describe("zmk,zkn->zmn", [24, 256, 256], [65536, 256, 1], [24, 256, 256], [65536, 256, 1])
    assert "resolve=fused" in desc, desc
    trop.reset_stats()
    rounds = 8
    for _ in range(rounds):
        for sr in SR:
            trop.gemm(dev[sr][0], dev[sr][1], sr, out=outs[sr][0], out_argmax=outs[sr][1])
    torch.cuda.synchronize()
    assert trop.stats()["gemm_early_starts"] >= rounds * 3 - 1
    for sr in SR:
        assert outs[sr][0].cpu().numpy().tobytes() == ref[sr][0].tobytes()
        np.testing.assert_array_equal(outs[sr][1].cpu().numpy(), ref[sr][1])


def test_gemm_reading_the_previous_output_waits_for_it(trop):
    """A GEMM whose operand is the previous GEMM's output must not start before that one has
    finished: no early start is counted for it, and the chain's result equals the oracle's."""
    a, b = _gemm_set(0)
    _, b2 = synth.gemm_batched_inputs(0, batch=24, m=256, n=256, k=256)
    ad, bd, b2d = _dev(a), _dev(b), _dev(b2[:, :, ::-1])
    c1, _ = trop.gemm(ad, bd, 0)
    trop.reset_stats()
    c2, i2 = trop.gemm(c1, b2d, 0)          # reads c1, written by the call just before
    torch.cuda.synchronize()
    assert trop.stats()["gemm_early_starts"] == 0
    rc1, _ = oracle.gemm(a, b, 0, nthreads=0)
    rc2, ri2 = oracle.gemm(rc1, np.ascontiguousarray(b2[:, :, ::-1]), 0, nthreads=0)
    assert c2.cpu().numpy().tobytes() == rc2.tobytes()
    np.testing.assert_array_equal(i2.cpu().numpy(), ri2)


def test_gemm_after_another_library_kernel_waits(trop):
    """A permute of this library between two GEMMs ends the chain: the second GEMM waits for
    the grid before it at its start (no early start), results exact."""
    a, b = _gemm_set(1)
    ad, bd = _dev(a), _dev(b)
    trop.gemm(ad, bd, 1)
    x = _dev(synth.uniform_f32(5, (64, 64), -1, 1))
    trop.permute_trace(x, "ij->ji")
    trop.reset_stats()
    c, i = trop.gemm(ad, bd, 1)
    torch.cuda.synchronize()
    assert trop.stats()["gemm_early_starts"] == 0
    rc, ri = oracle.gemm(a, b, 1, nthreads=0)
    assert c.cpu().numpy().tobytes() == rc.tobytes()
    np.testing.assert_array_equal(i.cpu().numpy(), ri)


@pytest.mark.parametrize("k", [16, 48, 64, 128, 256])
@pytest.mark.parametrize("sr", SR)
def test_one_launch_gemm_ragged_panels_and_short_k(trop, sr, k):
    """The one-launch GEMM + resolve on ragged shapes: 100 rows (one partial row block), 68
    columns (16-byte rows of B for TMA; a last panel of 4 columns), K from one 16-wide k-tile
    up, and enough tiles (80 batches x 4) that no tile is split along k.  Every output against
    the oracle."""
    bt, m, n = 80, 100, 68
    sa, sb = [bt, m, k], [bt, k, n]
    desc = trop.plan_describe("zmk,zkn->zmn", sa, [m * k, k, 1], sb, [k * n, n, 1])
    assert "kernel=tma" in desc and "resolve=fused" in desc, desc
    a, b = synth.gemm_batched_inputs(sr, batch=bt, m=m, n=n, k=k)
    _check(trop, a, b, sr)


def test_back_to_back_gemms_of_different_batch_counts(trop):
    """One-launch GEMMs of different batch counts, alternating on one stream and starting early
    behind each other: each keeps its own counters (the two halves of the stream's counters
    have a fixed layout), so every output equals the oracle's and no wait gives up."""
    shapes = [(0, 24, 256, 256, 256), (2, 80, 100, 68, 64), (1, 40, 192, 128, 128)]
    work = []
    for sr, bt, m, n, k in shapes:
        a, b = synth.gemm_batched_inputs(sr, batch=bt, m=m, n=n, k=k)
        rc, ri = oracle.gemm(a, b, sr, nthreads=0)
        outs = (torch.empty((bt, m, n), device="cuda"), torch.empty((bt, m, n), dtype=torch.int32, device="cuda"))
        work.append((sr, _dev(a), _dev(b), rc, ri, outs))
    trop.reset_stats()
    for rep in range(6):
        for j in ((0, 1, 2), (2, 0, 1), (1, 2, 0))[rep % 3]:
            sr, ad, bd, _, _, outs = work[j]
            trop.gemm(ad, bd, sr, out=outs[0], out_argmax=outs[1])
    torch.cuda.synchronize()
    trop.sync_pool()  # raises if a bounded wait gave up
    assert trop.stats()["gemm_early_starts"] >= 17
    for sr, ad, bd, rc, ri, outs in work:
        assert outs[0].cpu().numpy().tobytes() == rc.tobytes()
        np.testing.assert_array_equal(outs[1].cpu().numpy(), ri)


def test_random_mixed_gemm_sequences_stay_exact(trop):
    """Seeded random sequences of GEMM calls: mixed shapes and routes (one-launch GEMM at K = 256,
    64 and 16, the panel resolve at K = 1024, the cp.async tiles on ragged panels), with and
    without argmax, on two streams, into two output buffers per problem, half of them refilled
    first.  The last call on each buffer decides its contents, which must equal the oracle's
    bitwise.  This drives the early start of back-to-back one-launch GEMMs and the alternation
    of their counter halves through arbitrary interleavings."""
    import random
    probs = [(0, 64, 256, 256, 256), (1, 24, 256, 256, 256), (2, 80, 100, 68, 64), (0, 32, 256, 256, 1024),
             (1, 8, 128, 128, 64), (2, 80, 100, 68, 16), (0, 40, 192, 128, 128), (1, 6, 70, 45, 37)]
    data = []
    for sr, bt, m, n, k in probs:
        a, b = synth.gemm_batched_inputs(sr, batch=bt, m=m, n=n, k=k)
        rc, ri = oracle.gemm(a, b, sr, nthreads=0)
        outs = [(torch.empty((bt, m, n), device="cuda"), torch.empty((bt, m, n), dtype=torch.int32, device="cuda"))
                for _ in range(2)]
        data.append((sr, _dev(a), _dev(b), _dev(rc), _dev(ri), outs))
    streams = [torch.cuda.current_stream(), torch.cuda.Stream()]
    rng = random.Random(5)
    e0 = trop.stats()["gemm_early_starts"]
    bad = []
    for it in range(15):
        pending = []
        for _ in range(rng.randint(3, 12)):
            j = rng.randrange(len(data))
            sr, ad, bd, rc, ri, outs = data[j]
            o = rng.randrange(2)
            st = streams[1] if rng.random() < 0.3 else streams[0]
            if st is not streams[0]:
                st.wait_stream(streams[0])
            with torch.cuda.stream(st):
                if rng.random() < 0.5:
                    outs[o][0].fill_(0.0)
                    outs[o][1].fill_(-9)
                plain = rng.random() < 0.3
                if plain:
                    trop.gemm(ad, bd, sr, argmax=False, out=outs[o][0])
                else:
                    trop.gemm(ad, bd, sr, out=outs[o][0], out_argmax=outs[o][1])
            streams[0].wait_stream(st)
            pending.append((j, o, plain))
        torch.cuda.synchronize()
        seen = set()
        for j, o, plain in reversed(pending):
            if (j, o) in seen:
                continue
            seen.add((j, o))
            sr, ad, bd, rc, ri, outs = data[j]
            ok = torch.equal(outs[o][0].view(torch.int32), rc.view(torch.int32))
            if not plain:
                ok = ok and torch.equal(outs[o][1], ri)
            if not ok:
                bad.append((it, j, o, plain))
    trop.sync_pool()  # raises if a bounded wait gave up
    assert not bad, bad[:10]
    assert trop.stats()["gemm_early_starts"] > e0

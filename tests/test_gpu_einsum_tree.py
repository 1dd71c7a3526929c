"""GPU parity: pairwise einsum, contraction tree and back-tracking, workspace
pool behaviour, and error paths -- all through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def trop():
    import einsum_device_side_gb300 as t
    t.load()
    return t


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _cmp(trop, spec, a, b, sr=0, ad=None, bd=None):
    o, oa = trop.einsum(spec, _dev(a) if ad is None else ad, _dev(b) if bd is None else bd, sr)
    ro, roa = oracle.einsum(spec, a, b, sr, nthreads=0)
    assert o.cpu().numpy().tobytes() == ro.tobytes(), spec
    np.testing.assert_array_equal(oa.cpu().numpy(), roa, err_msg=spec)


@pytest.mark.parametrize("sr", [0, 1, 2])
def test_einsum_workload_reduced_size(trop, sr):
    lo = 0.0 if sr == 2 else -1.0
    A = synth.uniform_f32(1, (2, 64, 8, 8), lo, 1)
    B = synth.uniform_f32(2, (2, 8, 8, 72), lo, 1)
    _cmp(trop, "zacd,zdce->zea", A, B, sr)


def test_einsum_workload_full_size(trop):
    """'zacd,zdce->zea' at z=16, a=e=512, c=d=32 as benchmarked (B permuted,
    output transposed): every one of the 4,194,304 outputs' value and argmax
    bitwise against the oracle."""
    A, B = synth.einsum_inputs()
    o, oa = trop.einsum("zacd,zdce->zea", _dev(A), _dev(B))
    torch.cuda.synchronize()
    ro, roa = oracle.einsum("zacd,zdce->zea", A, B, nthreads=0)
    assert o.cpu().numpy().tobytes() == ro.tobytes()
    np.testing.assert_array_equal(oa.cpu().numpy(), roa)


@pytest.mark.parametrize("spec,sa,sb", [
    ("ij,jk->ik", (37, 23), (23, 41)),
    ("ij,jk->ki", (70, 33), (33, 90)),
    ("iij,jk->ik", (9, 9, 7), (7, 5)),            # diagonal in A
    ("ij,jk->k", (6, 8), (8, 5)),                  # one-operand label reduced first
    ("ijk,jkl->li", (5, 6, 7), (6, 7, 4)),         # two contracted labels, merged
    ("ikj,jkl->il", (5, 7, 6), (6, 7, 4)),         # contracted labels in swapped order: permute
    ("bij,bjk->bik", (3, 20, 30), (3, 30, 25)),
    ("bij,jk->bik", (3, 20, 30), (30, 25)),        # broadcast B over b
    ("ab,cd->abcd", (3, 4), (5, 2)),               # outer product, K = 1
    ("abc,cab->", (3, 4, 5), (5, 3, 4)),           # full contraction to a scalar
    ("zacd,zdce->zea", (2, 5, 3, 4), (2, 4, 3, 6)),
    ("xlub,lun->xlnb", (4, 2, 2, 8), (2, 2, 2)),   # the spin-glass step shape
    ("ab,ab->ab", (7, 9), (7, 9)),                 # elementwise (all batch)
    ("aij,jk->aik", (1, 13, 6), (6, 1)),           # unit extents
])
@pytest.mark.parametrize("sr", [0, 1, 2])
def test_einsum_specs(trop, spec, sa, sb, sr):
    lo = 0.0 if sr == 2 else -2.0
    a = np.round(synth.uniform_f32(21, sa, lo, 2) * 4) / 4          # coarse values: many ties
    b = np.round(synth.uniform_f32(22, sb, lo, 2) * 4) / 4
    _cmp(trop, spec, a.astype(np.float32), b.astype(np.float32), sr)


def test_einsum_strided_and_broadcast_operands(trop):
    a = synth.uniform_f32(3, (6, 40, 30), -1, 1)
    b = synth.uniform_f32(4, (30, 25), -1, 1)
    ad = _dev(a)[:, ::2, :]
    bd = _dev(b[None]).expand(3, 30, 25)
    _cmp(trop, "bij,bjk->bik", np.ascontiguousarray(a[:, ::2, :][:3]), np.broadcast_to(b[None], (3, 30, 25)), 0,
         ad[:3], bd)


def test_einsum_zero_extent(trop):
    a = torch.empty((3, 0), device="cuda")
    b = torch.empty((0, 4), device="cuda")
    o, oa = trop.einsum("ij,jk->ik", a, b, "maxplus")
    assert (o.cpu().numpy() == -np.inf).all() and (oa.cpu().numpy() == 0).all()


# ---------------------------------------------------------------- trees

def _ising(trop, rows, cols, seed):
    from einsum_device_side_gb300 import ising
    jh, jv = synth.couplings(seed, rows, cols)
    w, spins, _ = ising.ground_state(jh, jv)
    wo, so = oracle.ising_ground(jh, jv, rows, cols, nthreads=0)
    assert w == wo
    np.testing.assert_array_equal(spins, so)
    assert oracle.ising_energy(jh, jv, spins) == -w
    return jh, jv, w, spins


@pytest.mark.parametrize("rows,cols,seed", [(2, 2, 1), (4, 4, 2), (3, 7, 3), (8, 8, 4), (12, 10, 5)])
def test_ising_tree_matches_oracle(trop, rows, cols, seed):
    _ising(trop, rows, cols, seed)


def test_ising_workload_4x4_brute_force(trop):
    from einsum_device_side_gb300 import ising
    jh, jv = synth.ising_couplings(4, 4)
    w, spins, _ = ising.ground_state(jh, jv)
    wb, _ = oracle.ising_brute(jh, jv, 4, 4)
    assert w == wb and oracle.ising_energy(jh, jv, spins) == -w


def test_tree_unary_and_binary_nodes_generic(trop):
    # ((A x B) -> trace) with a diagonal input and an intermediate permute
    a = synth.uniform_f32(40, (5, 5, 6), -1, 1)
    b = synth.uniform_f32(41, (6, 7), -1, 1)
    c = synth.uniform_f32(42, (7, 3), -1, 1)
    I, J, K, L = 0, 1, 2, 3
    nodes = [(0, 1, [I, I, J], [J, K], [K, I]),      # 'iij,jk->ki'
             (3, None, [K, I], None, [I, K]),          # permute 'ki->ik'
             (4, 2, [I, K], [K, L], [I, L])]           # 'ik,kl->il'
    out = torch.empty((5, 3), device="cuda")
    am = [torch.empty((7, 5), dtype=torch.int32, device="cuda"), None,
          torch.empty((5, 3), dtype=torch.int32, device="cuda")]
    trop.contract_tree([_dev(a), _dev(b), _dev(c)], nodes, "maxplus", out, am)
    r1, ra1 = oracle.einsum("iij,jk->ki", a, b)
    r3, ra3 = oracle.einsum("ik,kl->il", np.ascontiguousarray(r1.T), c)
    np.testing.assert_array_equal(out.cpu().numpy(), r3)
    np.testing.assert_array_equal(am[0].cpu().numpy(), ra1)
    np.testing.assert_array_equal(am[2].cpu().numpy(), ra3)


def test_tree_rejects_bad_ids_before_launch(trop):
    a = torch.zeros((2, 2), device="cuda")
    with pytest.raises(trop.TropicalError) as e:
        trop.contract_tree([a], [(0, 5, [0, 1], [1, 2], [0, 2])], "maxplus", torch.empty((2, 2), device="cuda"))
    assert e.value.name == "INVALID_ARG"


# ---------------------------------------------------------------- pool

def test_pool_retires_through_events_without_stream_syncs(trop):
    trop.sync_pool()
    trop.reset_stats()
    trop.set_pool_capacity(1)          # force retirement pressure (the design note's "cache bound 1" test)
    try:
        for seed in (6, 7):
            _ising(trop, 5, 6, seed)
            a = synth.uniform_f32(seed, (3, 9, 8, 9), -1, 1)
            b = synth.uniform_f32(seed + 1, (8, 9, 9), -1, 1)
            _cmp(trop, "zikj,kij->zk", a, b)   # A's contracted labels are not adjacent: permuted in workspace
        s = trop.stats()
        assert s["pool_allocs"] > 0 and s["pool_retired"] > 0
        assert s["stream_syncs"] == 0
        trop.sync_pool()
        assert trop.stats()["stream_syncs"] == 0
    finally:
        trop.set_pool_capacity(16)


def test_pool_leaks_rather_than_races_on_event_failure(trop):
    trop.sync_pool()
    trop.reset_stats()
    trop.debug_fail_next_event_records(3)
    a = synth.uniform_f32(8, (3, 9, 8, 9), -1, 1)
    b = synth.uniform_f32(9, (8, 9, 9), -1, 1)
    _cmp(trop, "zikj,kij->zk", a, b)
    _cmp(trop, "zikj,kij->zk", a, b)
    s = trop.stats()
    assert s["pool_leaked"] >= 1
    trop.debug_fail_next_event_records(0)


def test_module_set_up_once(trop):
    before = trop.stats()["module_inits"]
    for _ in range(3):
        trop.gemm(torch.zeros((1, 8, 8), device="cuda"), torch.zeros((1, 8, 8), device="cuda"))
    assert trop.stats()["module_inits"] == before == 1


# ---------------------------------------------------------------- errors

def test_host_pointer_rejected(trop):
    with pytest.raises(trop.TropicalError) as e:
        trop.gemm(torch.zeros((1, 4, 4)), torch.zeros((1, 4, 4), device="cuda"))
    assert e.value.name == "HOST_POINTER"


def test_argmax_overflow_rejected(trop):
    a = torch.zeros((1, 1, 1), device="cuda").expand(1, 1, (1 << 31) + 1)
    b = torch.zeros((1, 1, 1), device="cuda").expand(1, (1 << 31) + 1, 1)
    with pytest.raises(trop.TropicalError) as e:
        trop.gemm(a, b, "maxplus")
    assert e.value.name == "OVERFLOW"


def test_spec_and_shape_errors(trop):
    a = torch.zeros((2, 3), device="cuda")
    with pytest.raises(trop.TropicalError) as e:
        trop.einsum("ij,jk->ik", a, torch.zeros((4, 5), device="cuda"))
    assert e.value.name == "SHAPE"
    with pytest.raises(trop.TropicalError) as e:
        trop.permute_trace(a, "ij->iq")
    assert e.value.name in ("SPEC",)
    with pytest.raises(trop.TropicalError) as e:
        trop.permute_trace(torch.zeros((2, 3), device="cuda"), "ii->i")
    assert e.value.name == "SHAPE"


def test_ising_workload_24x24_full_size(trop):
    """The benchmarked 24x24 instance: value and back-tracked configuration
    bitwise against the oracle's site-by-site elimination (OpenMP)."""
    from einsum_device_side_gb300 import ising
    jh, jv = synth.ising_couplings()
    w, spins, am = ising.ground_state(jh, jv)
    del am
    torch.cuda.empty_cache()
    wo, so = oracle.ising_ground(jh, jv, 24, 24, nthreads=0)
    assert w == wo
    np.testing.assert_array_equal(spins, so)
    assert oracle.ising_energy(jh, jv, spins) == -w


@pytest.mark.parametrize("rows,cols", [(8, 8), (5, 9)])
def test_ising_site_inputs_and_site_nodes_agree(trop, rows, cols):
    """The spin glass with its site tensors formed at build time (the default) and with one
    'ln,un->lun' node per site: the same value and back-tracked spins as the oracle."""
    from einsum_device_side_gb300 import ising
    jh, jv = synth.couplings(21, rows, cols)
    wo, so = oracle.ising_ground(jh, jv, rows, cols, nthreads=0)
    for site_nodes in (False, True):
        inputs, nodes, n_labels, need = ising.build_network(jh, jv, site_nodes=site_nodes)
        dev_in = [_dev(t) for t in inputs]
        am = [torch.empty([2] * len(nodes[j][4]), dtype=torch.int32, device="cuda") if j in need else None
              for j in range(len(nodes))]
        out = torch.empty((), device="cuda")
        trop.contract_tree(dev_in, nodes, "maxplus", out, am)
        assign = trop.tree_backtrack(dev_in, nodes, am, n_labels, 0)
        assert out.item() == wo
        np.testing.assert_array_equal(ising.spins_from_assignment(assign.cpu().numpy(), rows, cols), so)


# ---------------------------------------------------------------- plan cache

def test_plan_cache_lowers_a_repeated_einsum_once(trop):
    """A repeated pairwise einsum on tensors of the same layout is lowered once (the plan cache
    counts one miss, then hits) and its results stay bitwise equal to the oracle's; a change of
    layout (strides) is a new entry; disabling the cache lowers every call."""
    trop.set_plan_cache_capacity(64)
    A = synth.uniform_f32(61, (3, 40, 5, 6), -1, 1)
    B = synth.uniform_f32(62, (3, 6, 5, 33), -1, 1)
    ro, roa = oracle.einsum("zacd,zdce->zea", A, B, nthreads=0)
    Ad, Bd = _dev(A), _dev(B)
    s0 = trop.stats()
    for _ in range(5):
        o, oa = trop.einsum("zacd,zdce->zea", Ad, Bd)
        assert o.cpu().numpy().tobytes() == ro.tobytes()
        np.testing.assert_array_equal(oa.cpu().numpy(), roa)
    s1 = trop.stats()
    assert s1["plan_cache_misses"] - s0["plan_cache_misses"] == 1
    assert s1["plan_cache_hits"] - s0["plan_cache_hits"] == 4
    # a transposed view of B: another layout, another lowering, same values
    Bt = _dev(np.ascontiguousarray(np.transpose(B, (0, 3, 2, 1)))).permute(0, 3, 2, 1)
    o, oa = trop.einsum("zacd,zdce->zea", Ad, Bt)
    assert o.cpu().numpy().tobytes() == ro.tobytes()
    np.testing.assert_array_equal(oa.cpu().numpy(), roa)
    s2 = trop.stats()
    assert s2["plan_cache_misses"] - s1["plan_cache_misses"] == 1
    trop.set_plan_cache_capacity(0)
    try:
        for _ in range(2):
            o, oa = trop.einsum("zacd,zdce->zea", Ad, Bd)
        assert o.cpu().numpy().tobytes() == ro.tobytes()
        s3 = trop.stats()
        assert s3["plan_cache_hits"] == s2["plan_cache_hits"]
    finally:
        trop.set_plan_cache_capacity(64)


def test_plan_cache_evicts_least_recently_used(trop):
    """Beyond its bound the cache drops the least recently used layout: with a bound of 4,
    five distinct layouts in turn evict the first."""
    trop.set_plan_cache_capacity(4)
    try:
        ops = []
        for k in range(5):
            a = _dev(synth.uniform_f32(70 + k, (8, 9 + k), -1, 1))
            b = _dev(synth.uniform_f32(80 + k, (9 + k, 7), -1, 1))
            ops.append((a, b))
        for a, b in ops:
            trop.einsum("ij,jk->ik", a, b)
        s0 = trop.stats()
        trop.einsum("ij,jk->ik", *ops[4])          # most recent: a hit
        trop.einsum("ij,jk->ik", *ops[0])          # evicted: a miss
        s1 = trop.stats()
        assert s1["plan_cache_hits"] - s0["plan_cache_hits"] == 1
        assert s1["plan_cache_misses"] - s0["plan_cache_misses"] == 1
    finally:
        trop.set_plan_cache_capacity(64)


def test_tree_nodes_share_the_plan_cache(trop):
    """The contraction-tree executor lowers each node through the same cache: a second run
    of the 4x4 spin-glass tree lowers nothing and gives the same value."""
    from einsum_device_side_gb300 import ising
    trop.set_plan_cache_capacity(1024)
    try:
        jh, jv = synth.ising_couplings(4, 4)
        w0, _, _ = ising.ground_state(jh, jv, device="cuda")
        s0 = trop.stats()
        w1, _, _ = ising.ground_state(jh, jv, device="cuda")
        s1 = trop.stats()
        assert w1 == w0 == oracle.ising_ground(jh, jv, 4, 4)[0]
        assert s1["plan_cache_misses"] == s0["plan_cache_misses"]
        assert s1["plan_cache_hits"] > s0["plan_cache_hits"]
    finally:
        trop.set_plan_cache_capacity(64)

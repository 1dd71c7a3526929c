"""GPU parity of tree plans (tropical_tree_plan_*): a tree lowered once and
replayed as one CUDA graph must give exactly what the eager executor and the
oracle give, on every run, with inputs refilled in place between runs."""

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


def _ising_setup(rows, cols, seed):
    from einsum_device_side_gb300 import ising
    jh, jv = synth.couplings(seed, rows, cols)
    inputs, nodes, n_labels, need = ising.build_network(jh, jv)
    return jh, jv, inputs, nodes, n_labels, need


@pytest.mark.parametrize("rows,cols", [(4, 4), (8, 8), (12, 10)])
def test_ising_plan_matches_eager_and_oracle_across_refills(trop, rows, cols):
    from einsum_device_side_gb300 import ising
    jh, jv, inputs, nodes, n_labels, need = _ising_setup(rows, cols, 11)
    dev_in = [_dev(t) for t in inputs]
    out = torch.empty((), device="cuda")
    am = [torch.empty([2] * len(nodes[j][4]), dtype=torch.int32, device="cuda") if j in need else None
          for j in range(len(nodes))]
    plan = trop.tree_plan(dev_in, nodes, "maxplus", out, am)
    assert plan.kernels > 0 and plan.workspace_bytes > 0
    for rep, seed in enumerate([11, 12, 13, 11]):
        jh2, jv2, inputs2, nodes2, _, _ = _ising_setup(rows, cols, seed)
        assert [n[:2] for n in nodes2] == [n[:2] for n in nodes]          # same tree, new couplings
        for d, h in zip(dev_in, inputs2):
            d.copy_(torch.from_numpy(np.ascontiguousarray(h)))
        out.fill_(0)
        for a in am:
            if a is not None:
                a.fill_(-5)
        plan.run()
        # the eager executor on separate buffers
        out_e = torch.empty((), device="cuda")
        am_e = [torch.empty_like(a) if a is not None else None for a in am]
        trop.contract_tree(dev_in, nodes, "maxplus", out_e, am_e)
        torch.cuda.synchronize()
        assert out.item() == out_e.item()
        for a, b in zip(am, am_e):
            if a is not None:
                assert torch.equal(a, b)
        wo, so = oracle.ising_ground(jh2, jv2, rows, cols, nthreads=0)
        assert out.item() == wo
        assign = trop.tree_backtrack(dev_in, nodes, am, n_labels, 0)
        spins = ising.spins_from_assignment(assign.cpu().numpy(), rows, cols)
        assert oracle.ising_energy(jh2, jv2, spins) == -wo
    plan.close()


def test_generic_tree_plan_f32_and_f64(trop):
    I, J, K, L = 0, 1, 2, 3
    nodes = [(0, 1, [I, I, J], [J, K], [K, I]),      # 'iij,jk->ki'
             (3, None, [K, I], None, [I, K]),          # permute 'ki->ik'
             (4, 2, [I, K], [K, L], [I, L])]           # 'ik,kl->il'
    for dt, draw in ((torch.float32, synth.uniform_f32), (torch.float64, synth.uniform_f64)):
        a, b, c = draw(40, (5, 5, 6), -1, 1), draw(41, (6, 7), -1, 1), draw(42, (7, 3), -1, 1)
        ins = [_dev(a), _dev(b), _dev(c)]
        out = torch.empty((5, 3), dtype=dt, device="cuda")
        am = [torch.empty((7, 5), dtype=torch.int32, device="cuda"), None,
              torch.empty((5, 3), dtype=torch.int32, device="cuda")]
        plan = trop.tree_plan(ins, nodes, "maxplus", out, am)
        for _ in range(3):
            plan.run()
        torch.cuda.synchronize()
        r1, ra1 = oracle.einsum("iij,jk->ki", a, b)
        r3, ra3 = oracle.einsum("ik,kl->il", np.ascontiguousarray(r1.T), c)
        assert out.cpu().numpy().tobytes() == r3.tobytes()
        np.testing.assert_array_equal(am[0].cpu().numpy(), ra1)
        np.testing.assert_array_equal(am[2].cpu().numpy(), ra3)
        plan.close()


@pytest.mark.parametrize("sr", [0, 1, 2])
def test_single_node_plans_staging_permute_and_split_tail(trop, sr):
    """'zacd,zdce->zea' lowers to a B permute, a staged GEMM and a pair transpose;
    a plain batch-38 256^3 GEMM (no argmax) takes the stream-K tail, whose arrival
    counters the plan owns and zeroes by a captured memset."""
    lo = 0.0 if sr == 2 else -1.0
    A = synth.uniform_f32(1, (2, 64, 8, 8), lo, 1)
    B = synth.uniform_f32(2, (2, 8, 8, 72), lo, 1)
    Z, Aa, C, D, E = 0, 1, 2, 3, 4
    out = torch.empty((2, 72, 64), device="cuda")
    oam = torch.empty((2, 72, 64), dtype=torch.int32, device="cuda")
    plan = trop.tree_plan([_dev(A), _dev(B)], [(0, 1, [Z, Aa, C, D], [Z, D, C, E], [Z, E, Aa])], sr, out, [oam])
    plan.run()
    plan.run()
    ro, roa = oracle.einsum("zacd,zdce->zea", A, B, sr, nthreads=0)
    assert out.cpu().numpy().tobytes() == ro.tobytes()
    np.testing.assert_array_equal(oam.cpu().numpy(), roa)
    plan.close()
    a, b = synth.gemm_batched_inputs(sr, batch=38)
    ad, bd = _dev(a), _dev(b)
    ref = trop.gemm(ad, bd, sr, argmax=False)
    c = torch.empty_like(ref)
    plan = trop.tree_plan([ad, bd], [(0, 1, [0, 1, 2], [0, 2, 3], [0, 1, 3])], sr, c, None)
    for _ in range(3):
        c.fill_(0)
        plan.run()
        torch.cuda.synchronize()
        assert torch.equal(c, ref)
    plan.close()


def test_plan_counts_its_kernels_and_never_syncs(trop):
    jh, jv, inputs, nodes, n_labels, need = _ising_setup(6, 6, 3)
    dev_in = [_dev(t) for t in inputs]
    out = torch.empty((), device="cuda")
    plan = trop.tree_plan(dev_in, nodes, "maxplus", out, None)
    s0 = trop.stats()
    plan.run()
    plan.run()
    torch.cuda.synchronize()
    s1 = trop.stats()
    assert s1["kernel_launches"] - s0["kernel_launches"] == 2 * plan.kernels
    assert s1["stream_syncs"] == 0
    plan.close()
    plan.close()                       # idempotent


def test_plan_on_other_streams_and_errors(trop):
    jh, jv, inputs, nodes, n_labels, need = _ising_setup(5, 5, 4)
    dev_in = [_dev(t) for t in inputs]
    out = torch.empty((), device="cuda")
    plan = trop.tree_plan(dev_in, nodes, "maxplus", out, None)
    ref = torch.empty((), device="cuda")
    trop.contract_tree(dev_in, nodes, "maxplus", ref, None)
    for st in (torch.cuda.Stream(), torch.cuda.Stream()):
        out.fill_(0)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            plan.run()
        torch.cuda.synchronize()
        assert out.item() == ref.item()
    plan.close()
    with pytest.raises(RuntimeError):
        plan.run()
    a = torch.zeros((2, 2), device="cuda")
    with pytest.raises(trop.TropicalError):
        trop.tree_plan([a], [(0, 5, [0, 1], [1, 2], [0, 2])], "maxplus", torch.empty((2, 2), device="cuda"))

"""The spin-glass network builder (host logic, no GPU): both forms of the tree -- site tensors
formed at build time, or one 'ln,un->lun' node per site -- evaluated node by node with the CPU
oracle's einsum give the ground-state value of the oracle's elimination and of brute force."""
import numpy as np
import pytest

import oracle
import synth
from einsum_device_side_gb300 import ising


def _labels(ls):
    return "".join(chr(97 + x) if x < 26 else chr(65 + x - 26) for x in ls)


def _evaluate(inputs, nodes):
    vals = list(inputs)
    for a, b, la, lb, lo in nodes:
        if b is None:
            v, _ = oracle.einsum(_labels(la) + "->" + _labels(lo), vals[a], nthreads=0)
        else:
            v, _ = oracle.einsum(_labels(la) + "," + _labels(lb) + "->" + _labels(lo), vals[a], vals[b], nthreads=0)
        vals.append(v)
    return float(vals[-1])


@pytest.mark.parametrize("rows,cols,seed", [(2, 2, 1), (3, 4, 2), (4, 4, 3), (4, 3, 4)])
def test_both_tree_forms_give_the_ground_state(rows, cols, seed):
    jh, jv = synth.couplings(seed, rows, cols)
    wb, _ = oracle.ising_brute(jh, jv, rows, cols)
    for site_nodes in (False, True):
        inputs, nodes, n_labels, need = ising.build_network(jh, jv, site_nodes=site_nodes)
        assert n_labels == rows * cols
        assert _evaluate(inputs, nodes) == wb


def test_site_tensor_is_the_sum_of_its_two_bonds():
    for jl in (-1, 1):
        for ju in (-1, 1):
            q = ising.site(jl, ju)
            s = np.array([-1, 1])
            want = jl * s[:, None, None] * s[None, None, :] + ju * s[None, :, None] * s[None, None, :]
            np.testing.assert_array_equal(q, want.astype(np.float32))


def test_tree_sizes_of_the_24x24_workload():
    jh, jv = synth.ising_couplings()
    inputs, nodes, _, need = ising.build_network(jh, jv)
    # 22 row-0 steps, 23 x 24 contracting steps, the final reduction
    assert len(nodes) == 22 + 552 + 1 and len(need) == 553
    inputs2, nodes2, _, need2 = ising.build_network(jh, jv, site_nodes=True)
    assert len(nodes2) == len(nodes) + 23 * 23 and len(need2) == 553

"""Open-boundary 2-D spin glass as a max-plus contraction tree.

The ground state of H = -sum J_ij s_i s_j (zero field, couplings on the
nearest-neighbour bonds of an R x C grid) is W = max over spins of
sum J s_i s_j, E0 = -W.  In max-plus algebra W is the contraction of one
2x2 bond tensor T[x, y] = J * s(x) * s(y), s(x) = 2x - 1, per bond.

Tree (labels: spin (r, c) -> r*C + c):
  * row 0: the first bond is the initial frontier; each further site of the
    row appends its spin:  'X l, l n -> X l n' (no contraction).
  * each site (r, c), r >= 1: the frontier spin u = (r-1, c) is contracted
    with the site tensor Q[l, u, n] = T_left[l, n] + T_up[u, n]:
    'X l u Y, l u n -> X l n Y' (for c = 0 only the up bond: 'u Y, u n -> n Y').
    Q depends on two couplings only, so it is formed with the bond tensors
    when the network is built (2 x 2 x 2, sums of +-1: exact); with
    site_nodes=True it is a tree node of its own instead ('ln,un->lun', n
    shared), one small kernel per site.
  * a final trace reduces the whole last row:  'f0 .. f_{C-1} ->' with argmax.
The frontier always holds one spin per column (2**C entries).  The argmax of
each contraction node records the winning u; back-tracking from the final
argmax through them recovers an optimal configuration.
"""

from __future__ import annotations

import numpy as np


def bond(j: int) -> np.ndarray:
    s = np.array([-1.0, 1.0], dtype=np.float32)
    return (float(j) * s[:, None] * s[None, :]).astype(np.float32)


def site(jl: int, ju: int) -> np.ndarray:
    """Q[l, u, n] = T_left[l, n] + T_up[u, n] (float32, exact)."""
    return (bond(jl)[:, None, :] + bond(ju)[None, :, :]).astype(np.float32)


def build_network(jh: np.ndarray, jv: np.ndarray, site_nodes: bool = False):
    """Returns (inputs, nodes, n_labels, contraction_nodes).

    inputs: list of float32 numpy arrays (bond tensors);
    nodes: list of (lhs, rhs, lhs_labels, rhs_labels, out_labels);
    contraction_nodes: indices of nodes whose argmax is needed for
    back-tracking (the up-spin contractions and the final trace)."""
    R, C = jh.shape[0], jh.shape[1] + 1
    assert jv.shape == (R - 1, C) and R >= 2 and C >= 2
    lab = lambda r, c: r * C + c  # noqa: E731
    inputs, nodes, need = [], [], []

    def add_input(t):
        inputs.append(t)
        return len(inputs) - 1

    # placeholders: node ids are offsets by the final number of inputs, so
    # collect (kind, payload) first and resolve ids at the end
    ops = []
    first = add_input(bond(jh[0, 0]))
    state = ("in", first)
    front = [lab(0, 0), lab(0, 1)]
    for c in range(2, C):
        t = add_input(bond(jh[0, c - 1]))
        out = front + [lab(0, c)]
        ops.append((state, ("in", t), list(front), [lab(0, c - 1), lab(0, c)], out, False))
        state = ("node", len(ops) - 1)
        front = out
    for r in range(1, R):
        for c in range(C):
            u, n = lab(r - 1, c), lab(r, c)
            out = list(front)
            out[c] = n
            if c == 0:
                tu = add_input(bond(jv[r - 1, c]))
                ops.append((state, ("in", tu), list(front), [u, n], out, True))
            else:
                l = lab(r, c - 1)
                if site_nodes:
                    tu = add_input(bond(jv[r - 1, c]))
                    tl = add_input(bond(jh[r, c - 1]))
                    ops.append((("in", tl), ("in", tu), [l, n], [u, n], [l, u, n], False))
                    q = ("node", len(ops) - 1)
                else:
                    q = ("in", add_input(site(jh[r, c - 1], jv[r - 1, c])))
                ops.append((state, q, list(front), [l, u, n], out, True))
            state = ("node", len(ops) - 1)
            front = out
    ops.append((state, None, list(front), None, [], True))
    nin = len(inputs)

    def rid(x):
        if x is None:
            return None
        kind, i = x
        return i if kind == "in" else nin + i

    for j, (a, b, la, lb, lo, needs) in enumerate(ops):
        nodes.append((rid(a), rid(b), la, lb, lo))
        if needs:
            need.append(j)
    return inputs, nodes, R * C, need


def spins_from_assignment(assign: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """label values (0/1) -> spins (+-1), shape (rows, cols)."""
    a = np.asarray(assign).reshape(rows, cols)
    if (a < 0).any():
        raise ValueError("back-tracking left spins undetermined")
    return (2 * a - 1).astype(np.int8)


def energy(jh: np.ndarray, jv: np.ndarray, spins: np.ndarray) -> int:
    s = spins.astype(np.int64)
    return int(-(jh * s[:, :-1] * s[:, 1:]).sum() - (jv * s[:-1, :] * s[1:, :]).sum())


def ground_state(jh, jv, device="cuda", keep_argmax=True, site_nodes=False):
    """Contract the network on the GPU; returns (W, spins, per-node argmax).

    W = max sum J s s (E0 = -W).  site_nodes: as in build_network."""
    import torch

    from . import contract_tree, tree_backtrack

    inputs, nodes, n_labels, need = build_network(jh, jv, site_nodes=site_nodes)
    dev_inputs = [torch.from_numpy(t).to(device) for t in inputs]
    R, C = jh.shape[0], jh.shape[1] + 1
    out = torch.empty((), dtype=torch.float32, device=device)
    am = [None] * len(nodes)
    if keep_argmax:
        for j in need:
            shape = [2] * len(nodes[j][4])
            am[j] = torch.empty(shape, dtype=torch.int32, device=device)
    contract_tree(dev_inputs, nodes, "maxplus", out, am)
    spins = None
    if keep_argmax:
        assign = tree_backtrack(dev_inputs, nodes, am, n_labels, 0)
        spins = spins_from_assignment(assign.cpu().numpy(), R, C)
    return float(out.item()), spins, am

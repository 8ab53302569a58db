"""Pins for the float64 oracle: each check ties it to something other than itself.

The gated delta rule and the tree semantics come from "Trees from Marginals"
(gist.science Technical Summary, section 3 "Rollback-Free Tree Verification for
GDN").  The pins:
  * hand-worked values on tiny trees (tests/golden/scalar_tree.txt);
  * the delta-rule write property: beta = 1, |k| = 1, q = k gives o_i = v_i;
  * the beta = 0 closed form o_i = exp(gamma_i) S0 q_i, with ancestors from networkx;
  * brute force over every forest with N <= 6 against the matrix form of the
    same section (interaction matrices X, Y and the linear system
    (I + X) U = R), solved with numpy.linalg.solve;
  * a 64-node chain against the same matrix form;
  * sibling independence, relabelling invariance, linearity in (S0, V);
  * commit = walked state, and chain composition through a commit;
  * the descriptor against networkx ancestors and depths.
"""
import itertools
import math
import os

import networkx as nx
import numpy as np
import pytest

import oracle
from gated_delta_net_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scalar_tree.txt")


def _tb_from_arrays(parent, q, k, v, g, beta, S0, Hk=1, Hv=1, scale=1.0, paths=None):
    parent = np.asarray(parent, np.int32)
    n = len(parent)
    dk, dv = k.shape[-1], v.shape[-1]
    tb = W.TreeBatch("t", 1, Hk, Hv, dk, dv, "f32", np.array([0, n], np.int32), parent,
                     np.asarray(q, np.float64).reshape(n, Hk, dk),
                     np.asarray(k, np.float64).reshape(n, Hk, dk),
                     np.asarray(v, np.float64).reshape(n, Hv, dv),
                     np.asarray(g, np.float64).reshape(n, Hv),
                     np.asarray(beta, np.float64).reshape(n, Hv),
                     np.asarray(S0, np.float64).reshape(1, Hv, dv, dk),
                     np.array([0, 0], np.int32), np.zeros(0, np.int32), scale)
    if paths is not None:
        tb.path_offsets = np.array([0, len(paths)], np.int32)
        tb.path_idx = np.asarray(paths, np.int32)
    return tb


def _random_tb(rng, parent, dk=3, dv=2, Hk=1, Hv=1, beta=None, qk_same=False):
    n = len(parent)
    k = rng.standard_normal((n, Hk, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q = k.copy() if qk_same else rng.standard_normal((n, Hk, dk))
    v = rng.standard_normal((n, Hv, dv))
    g = -np.log1p(np.exp(rng.standard_normal((n, Hv))))
    b = rng.uniform(0.05, 0.95, (n, Hv)) if beta is None else np.full((n, Hv), beta)
    S0 = 0.3 * rng.standard_normal((1, Hv, dv, dk))
    return _tb_from_arrays(parent, q, k, v, g, b, S0, Hk, Hv)


def _ancestors(parent):
    """Inclusive ancestor sets via networkx (independent of the oracle's walk)."""
    G = nx.DiGraph()
    G.add_nodes_from(range(len(parent)))
    G.add_edges_from((int(p), i) for i, p in enumerate(parent) if p >= 0)
    return [nx.ancestors(G, i) | {i} for i in range(len(parent))]


def _matrix_form(tb, h=0):
    """Outputs and per-node states from the interaction-matrix form.

    gamma_i = sum of g over anc(i); D_ij = exp(gamma_i - gamma_j) for j in anc(i);
    X_ij = beta_i D_ij (k_i . k_j) on strict ancestors; Y_ij = D_ij (q_i . k_j) on
    inclusive ancestors; R = beta * (V - exp(gamma) * K S0^T);
    U = solve(I + X, R);  O = exp(gamma) * Q S0^T + Y U;
    S_i = exp(gamma_i) S0 + sum_{j in anc(i)} D_ij u_j k_j^T.
    """
    parent = tb.parent
    n = len(parent)
    anc = _ancestors(parent)
    hk = h // (tb.n_v_heads // tb.n_k_heads)
    K, Q = tb.k[:, hk, :].astype(np.float64), tb.q[:, hk, :].astype(np.float64)
    V = tb.v[:, h, :].astype(np.float64)
    g, beta = tb.g[:, h].astype(np.float64), tb.beta[:, h].astype(np.float64)
    S0 = tb.S0[0, h].astype(np.float64)
    gam = np.array([sum(g[j] for j in anc[i]) for i in range(n)])
    X = np.zeros((n, n))
    Y = np.zeros((n, n))
    for i in range(n):
        for j in anc[i]:
            D = math.exp(gam[i] - gam[j])
            Y[i, j] = D * Q[i] @ K[j]
            if j != i:
                X[i, j] = beta[i] * D * K[i] @ K[j]
    R = beta[:, None] * (V - np.exp(gam)[:, None] * (K @ S0.T))
    U = np.linalg.solve(np.eye(n) + X, R)
    O = np.exp(gam)[:, None] * (Q @ S0.T) + Y @ U
    S = [np.exp(gam[i]) * S0 + sum(math.exp(gam[i] - gam[j]) * np.outer(U[j], K[j])
                                   for j in anc[i]) for i in range(n)]
    return tb.scale * O, S


# ----------------------------------------------------------------------------
# hand-worked golden values
# ----------------------------------------------------------------------------

def _parse_golden(path):
    cases, cur = [], None
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        tok = line.split()
        if tok[0] == "case":
            cur = {"name": tok[1], "dk": int(tok[2][3:]), "dv": int(tok[3][3:]),
                   "nodes": [], "expect": {}}
        elif tok[0] == "S0":
            cur["S0"] = [float(x) for x in tok[1:]]
        elif tok[0] == "node":
            cur["nodes"].append([float(x) for x in tok[1:]])
        elif tok[0] == "expect":
            cur["expect"][int(tok[1])] = [float(x) for x in tok[2:]]
        elif tok[0] == "end":
            cases.append(cur)
    return cases


@pytest.mark.parametrize("case", _parse_golden(GOLDEN), ids=lambda c: c["name"])
def test_hand_worked_values(case):
    dk, dv = case["dk"], case["dv"]
    nodes = sorted(case["nodes"], key=lambda r: r[0])
    parent = [int(r[1]) for r in nodes]
    alpha = np.array([r[2] for r in nodes])
    beta = np.array([r[3] for r in nodes])
    k = np.array([r[4:4 + dk] for r in nodes])
    v = np.array([r[4 + dk:4 + dk + dv] for r in nodes])
    q = np.array([r[4 + dk + dv:4 + 2 * dk + dv] for r in nodes])
    tb = _tb_from_arrays(parent, q, k, v, np.log(alpha), beta, np.array(case["S0"]))
    o = oracle.verify(tb)[:, 0, :]
    for i, exp in case["expect"].items():
        np.testing.assert_allclose(o[i], exp, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(4))
def test_delta_rule_write_property(seed):
    """beta = 1, unit k, q = k: S_i k_i = v_i, so o_i = v_i on every tree."""
    rng = np.random.default_rng(seed)
    parent = W.uniform_recursive_tree(rng, 20)
    tb = _random_tb(rng, parent, dk=5, dv=4, Hk=2, Hv=4, beta=1.0, qk_same=True)
    o = oracle.verify(tb)
    np.testing.assert_allclose(o, tb.v, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_beta_zero_closed_form(seed):
    rng = np.random.default_rng(seed)
    parent = W.depth_capped_random_tree(rng, 25, max_depth=6)
    tb = _random_tb(rng, parent, dk=4, dv=3, beta=0.0)
    tb.scale = 0.75
    anc = _ancestors(parent)
    o = oracle.verify(tb)[:, 0, :]
    for i in range(len(parent)):
        gam = sum(tb.g[j, 0] for j in anc[i])
        np.testing.assert_allclose(o[i], 0.75 * math.exp(gam) * tb.S0[0, 0] @ tb.q[i, 0],
                                   rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------
# brute force against the matrix form
# ----------------------------------------------------------------------------

def _all_forests(n):
    for choice in itertools.product(*[range(-1, i) for i in range(n)]):
        yield np.array(choice, np.int32)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_brute_force_all_forests(n):
    rng = np.random.default_rng(100 + n)
    count = 0
    for parent in _all_forests(n):
        tb = _random_tb(rng, parent, dk=3, dv=2)
        o = oracle.verify(tb)[:, 0, :]
        O, S = _matrix_form(tb)
        np.testing.assert_allclose(o, O, rtol=1e-10, atol=1e-12)
        # every node's walked state equals the matrix-form state; commit every leaf path
        for i in range(n):
            np.testing.assert_allclose(oracle.state_at(tb, 0, 0, i), S[i], rtol=1e-10,
                                       atol=1e-12)
        count += 1
    assert count == math.factorial(n)


def test_brute_force_commit_every_leaf():
    rng = np.random.default_rng(7)
    for parent in _all_forests(5):
        tb = _random_tb(rng, parent, dk=2, dv=3)
        _, S = _matrix_form(tb)
        has_child = set(int(p) for p in parent if p >= 0)
        for leaf in range(len(parent)):
            if leaf in has_child:
                continue
            path = []
            j = leaf
            while j >= 0:
                path.append(j)
                j = int(parent[j])
            tb.path_offsets = np.array([0, len(path)], np.int32)
            tb.path_idx = np.array(path[::-1], np.int32)
            Snew, st = oracle.commit(tb)
            assert st == 0
            np.testing.assert_allclose(Snew[0, 0], S[leaf], rtol=1e-10, atol=1e-12)


def test_chain_matches_matrix_form():
    rng = np.random.default_rng(11)
    tb = _random_tb(rng, W.chain_tree(64), dk=16, dv=8)
    O, _ = _matrix_form(tb)
    np.testing.assert_allclose(oracle.verify(tb)[:, 0, :], O, rtol=1e-9, atol=1e-11)


def test_head_sharing_equals_duplicated_key_heads():
    """Value head h reads key head h // (Hv / Hk)."""
    rng = np.random.default_rng(5)
    parent = W.uniform_recursive_tree(rng, 10)
    tb = _random_tb(rng, parent, dk=3, dv=3, Hk=2, Hv=4)
    dup = _random_tb(rng, parent, dk=3, dv=3, Hk=4, Hv=4)
    dup.q = tb.q[:, [0, 0, 1, 1], :].copy()
    dup.k = tb.k[:, [0, 0, 1, 1], :].copy()
    dup.v, dup.g, dup.beta, dup.S0 = tb.v, tb.g, tb.beta, tb.S0
    np.testing.assert_array_equal(oracle.verify(tb), oracle.verify(dup))
    for h in range(4):
        O, _ = _matrix_form(tb, h)
        np.testing.assert_allclose(oracle.verify(tb)[:, h, :], O, rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------------------
# structural invariants
# ----------------------------------------------------------------------------

def test_sibling_independence_bit_exact():
    rng = np.random.default_rng(3)
    parent = W.depth_capped_random_tree(rng, 30, max_depth=8)
    tb = _random_tb(rng, parent, dk=4, dv=4)
    base = oracle.verify(tb)
    anc = _ancestors(parent)
    target = 17
    outside = [j for j in range(30) if j not in anc[target]]
    for bad in (np.nan, np.inf, -np.inf, 1e30):
        tb2 = _random_tb(rng, parent, dk=4, dv=4)
        tb2.q, tb2.k, tb2.v = tb.q.copy(), tb.k.copy(), tb.v.copy()
        tb2.g, tb2.beta, tb2.S0 = tb.g.copy(), tb.beta.copy(), tb.S0
        tb2.k[outside] = bad
        tb2.v[outside] = bad
        tb2.g[outside] = bad
        o2 = oracle.verify(tb2)
        for i in range(30):
            if set(anc[i]).isdisjoint(outside):
                np.testing.assert_array_equal(o2[i], base[i])


def test_relabelling_permutes_outputs():
    rng = np.random.default_rng(9)
    parent = W.depth_capped_random_tree(rng, 24, max_depth=7)
    tb = _random_tb(rng, parent, dk=3, dv=3)
    # another topological order: BFS by depth, children visited in reverse order
    children = {i: [] for i in range(24)}
    for i, p in enumerate(parent):
        if p >= 0:
            children[int(p)].append(i)
    order, frontier = [], [i for i in range(24) if parent[i] < 0]
    while frontier:
        order += frontier
        frontier = [c for f in frontier for c in reversed(children[f])]
    new_of = {old: new for new, old in enumerate(order)}
    perm = np.array(order)
    parent2 = np.array([new_of[int(parent[o])] if parent[o] >= 0 else -1 for o in order],
                       np.int32)
    assert all(parent2[i] < i for i in range(24))
    tb2 = _tb_from_arrays(parent2, tb.q[perm], tb.k[perm], tb.v[perm], tb.g[perm],
                          tb.beta[perm], tb.S0)
    np.testing.assert_array_equal(oracle.verify(tb2), oracle.verify(tb)[perm])


def test_linear_in_state_and_values():
    rng = np.random.default_rng(13)
    parent = W.uniform_recursive_tree(rng, 15)
    a = _random_tb(rng, parent, dk=4, dv=3)
    b = _random_tb(rng, parent, dk=4, dv=3)
    b.q, b.k, b.g, b.beta = a.q, a.k, a.g, a.beta
    c = _random_tb(rng, parent, dk=4, dv=3)
    c.q, c.k, c.g, c.beta = a.q, a.k, a.g, a.beta
    c.v = 2.0 * a.v - 3.0 * b.v
    c.S0 = 2.0 * a.S0 - 3.0 * b.S0
    np.testing.assert_allclose(oracle.verify(c), 2 * oracle.verify(a) - 3 * oracle.verify(b),
                               rtol=1e-10, atol=1e-12)


def test_scale_multiplies_outputs():
    rng = np.random.default_rng(17)
    tb = _random_tb(rng, W.uniform_recursive_tree(rng, 9), dk=3, dv=3)
    o1 = oracle.verify(tb)
    tb.scale = 0.125
    np.testing.assert_allclose(oracle.verify(tb), 0.125 * o1, rtol=1e-14, atol=0)


# ----------------------------------------------------------------------------
# commit
# ----------------------------------------------------------------------------

def test_commit_readout_equals_verify_output():
    tb = W.tiny_tree(0)
    o = oracle.verify(tb)
    S, st = oracle.commit(tb)
    assert st == 0
    leaf = int(tb.path_idx[-1])
    np.testing.assert_allclose(S[0, 0] @ tb.q[leaf, 0].astype(np.float64), o[leaf, 0],
                               rtol=1e-12, atol=1e-14)


def test_chain_composition_through_commit():
    """Verifying a chain's tail from the committed prefix state equals the tail of
    verifying the whole chain (the delayed commit of the same section)."""
    rng = np.random.default_rng(21)
    tb = _random_tb(rng, W.chain_tree(20), dk=4, dv=5, Hk=1, Hv=2)
    full = oracle.verify(tb)
    split = 8
    tb.path_offsets = np.array([0, split], np.int32)
    tb.path_idx = np.arange(split, dtype=np.int32)
    S_mid, st = oracle.commit(tb)
    assert st == 0
    tail = _tb_from_arrays(W.chain_tree(20 - split), tb.q[split:], tb.k[split:], tb.v[split:],
                           tb.g[split:], tb.beta[split:], S_mid, Hk=1, Hv=2)
    np.testing.assert_allclose(oracle.verify(tail), full[split:], rtol=1e-11, atol=1e-13)


def test_commit_rejects_bad_paths():
    tb = W.tiny_tree(0)
    for bad in ([1], [0, 0], [0, 99], [-1]):
        _, st = oracle.commit(tb, path_offsets=[0, len(bad)], path_idx=bad)
        assert st == 2
    S, st = oracle.commit(tb, path_offsets=[0, 0], path_idx=[])
    assert st == 0
    np.testing.assert_array_equal(S, tb.S0)


# ----------------------------------------------------------------------------
# descriptor
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("maker", ["uniform", "capped", "best_first", "chain"])
def test_descriptor_against_networkx(maker):
    rng = np.random.default_rng(31)
    parents = []
    for n in (1, 2, 31, 32, 33, 64, 100, 128):
        if maker == "uniform":
            parents.append(W.uniform_recursive_tree(rng, n))
        elif maker == "capped":
            parents.append(W.depth_capped_random_tree(rng, n))
        elif maker == "best_first":
            parents.append(W.best_first_tree(rng, n))
        else:
            parents.append(W.chain_tree(n))
    offsets = np.concatenate([[0], np.cumsum([len(p) for p in parents])]).astype(np.int32)
    mask, depth, st = oracle.build_desc(np.concatenate(parents), offsets, 4)
    assert st == 0
    for b, parent in enumerate(parents):
        anc = _ancestors(parent)
        for i in range(len(parent)):
            row = mask[offsets[b] + i]
            bits = {w * 32 + j for w in range(4) for j in range(32) if (int(row[w]) >> j) & 1}
            assert bits == anc[i]
            assert depth[offsets[b] + i] == len(anc[i])


def test_descriptor_flags_bad_parent():
    for parent in ([0], [-1, 1], [-1, 0, 5], [-1, -2]):
        _, _, st = oracle.build_desc(np.array(parent, np.int32),
                                     np.array([0, len(parent)], np.int32), 1)
        assert st == 1


# ----------------------------------------------------------------------------
# selected outputs (the checker of the full-size GPU tests and the CPU baseline)
# ----------------------------------------------------------------------------

def _selection_batch(kind):
    """Ragged multi-request batches for the selected-output oracle.

    "square": every request has exactly Hv nodes (3 requests, Hk = 2, Hv = 4,
    d_k = 3, d_v = 5), so any (h, i) mix-up stays inside the arrays.
    "ragged": sizes 3, 0, 7, 1, 0, 5 (empty requests and forests), Hk = 2, Hv = 4,
    d_k = 3, d_v = 5.  "wide": 16 key / 32 value heads, d_k = 8, d_v = 6, sizes 5, 0, 9.
    """
    rng = np.random.default_rng({"square": 41, "ragged": 42, "wide": 43}[kind])
    if kind == "square":
        sizes, Hk, Hv, dk, dv = [4, 4, 4], 2, 4, 3, 5
    elif kind == "ragged":
        sizes, Hk, Hv, dk, dv = [3, 0, 7, 1, 0, 5], 2, 4, 3, 5
    else:
        sizes, Hk, Hv, dk, dv = [5, 0, 9], 16, 32, 8, 6
    parents = []
    for n in sizes:
        # forests: every node after the first is a root with probability 1/4
        par = np.array([-1 if i == 0 or rng.random() < 0.25 else int(rng.integers(0, i))
                        for i in range(n)], np.int32)
        parents.append(par)
    tb = W.make_batch("sel_" + kind, 7, parents, Hk, Hv, dk, dv, "f32", W.path_random_leaf)
    return tb


@pytest.mark.parametrize("kind", ["square", "ragged", "wide"])
def test_verify_selected_matches_verify(kind):
    """oracle.verify_selected(tb, sel)[r] equals oracle.verify(tb)[offsets[b] + i, h]
    bit for bit for every selected (b, h, i): exhaustively, and for a random
    selection with repeats in random order."""
    tb = _selection_batch(kind)
    full = oracle.verify(tb)
    offs = tb.node_offsets
    sel = [(b, h, i) for b in range(tb.batch) for h in range(tb.n_v_heads)
           for i in range(int(offs[b + 1] - offs[b]))]
    rng = np.random.default_rng(5)
    rand = [sel[j] for j in rng.integers(0, len(sel), 3 * len(sel))]
    for chosen in (sel, rand):
        got = oracle.verify_selected(tb, chosen, nthreads=3)
        want = np.stack([full[offs[b] + i, h] for b, h, i in chosen])
        np.testing.assert_array_equal(got, want)

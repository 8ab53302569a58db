"""Pins for the topological-relabel oracle (oracle/relabel.py).

The requirement comes from "Trees from Marginals" (gist.science Technical
Summary, section 3, Solution, bullet 1): nodes are processed in topological
order.  The relabel order is (depth, old id).  It is pinned here to something
other than the oracle's own parent walk:
  * networkx's topological generations of the same forest (generation g holds
    the nodes of depth g + 1), each generation sorted by id, for every forest
    with N <= 6 under several random relabellings;
  * the relabelled forest is the same forest: parent_out[rank[i]] = rank[parent[i]];
  * closed forms: a chain labelled backwards comes out reversed; an already
    depth-sorted tree is the identity;
  * malformed arrays (a cycle, a self-parent, a parent out of range) are flagged.
"""
import itertools

import networkx as nx
import numpy as np
import pytest

from oracle import relabel as R


def _generations_order(parent):
    g = nx.DiGraph()
    g.add_nodes_from(range(len(parent)))
    g.add_edges_from((int(p), i) for i, p in enumerate(parent) if p >= 0)
    return [i for gen in nx.topological_generations(g) for i in sorted(gen)]


def _forests(n):
    return itertools.product(*[range(-1, i) for i in range(n)])


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_every_forest_under_random_labellings(n):
    rng = np.random.default_rng(n)
    for par in _forests(n):
        par = np.array(par, np.int64)
        for _ in range(3):
            perm = rng.permutation(n)          # old label i -> new label perm[i]
            shuffled = np.empty(n, np.int64)
            for i in range(n):
                shuffled[perm[i]] = -1 if par[i] < 0 else perm[par[i]]
            order, rank, parent_out = R.relabel_one(shuffled)
            assert list(order) == _generations_order(shuffled)
            assert sorted(order) == list(range(n))
            assert all(rank[order[j]] == j for j in range(n))
            assert all(parent_out[j] < j for j in range(n))
            for i in range(n):
                want = -1 if shuffled[i] < 0 else rank[shuffled[i]]
                assert parent_out[rank[i]] == want


def test_backwards_chain_comes_out_reversed():
    n = 9
    parent = np.array([i + 1 for i in range(n - 1)] + [-1])   # node n-1 is the root
    order, rank, parent_out = R.relabel_one(parent)
    assert list(order) == list(range(n - 1, -1, -1))
    assert list(parent_out) == [-1] + list(range(n - 1))


def test_depth_sorted_tree_is_identity():
    parent = np.array([-1, 0, 0, 1, 1, 2, 3, -1, 7])
    # depths: 1, 2, 2, 3, 3, 3, 4, 1, 2 -> not depth-sorted; sort it first
    order, _, parent_out = R.relabel_one(parent)
    o2, r2, p2 = R.relabel_one(parent_out)
    assert list(o2) == list(range(len(parent)))
    assert list(p2) == list(parent_out)


@pytest.mark.parametrize("parent", [[1, 0], [0], [-1, 5], [-2, 0], [-1, 2, 1], [-1, 0, 3, 2]])
def test_malformed_arrays_are_flagged(parent):
    assert R.relabel_one(np.array(parent)) is None
    order, rank, parent_out, bad = R.relabel(np.array(parent + [-1, 0]), np.array([0, len(parent), len(parent) + 2]))
    assert bad.tolist() == [True, False]
    assert order[-2:].tolist() == [0, 1]


@pytest.mark.parametrize("mutant", ["no_depth_key", "ties_descending", "old_id_parents", "depth_off_by_one_root"])
def test_pins_catch_planted_mistakes(mutant, monkeypatch):
    # each mutant is a plausible slip in the oracle; one of the pins above must fail
    real_one, real_depths = R.relabel_one, R.depths

    def mutated(parent):
        parent = np.asarray(parent, np.int64)
        dep = real_depths(parent)
        if dep is None:
            return None
        n = len(parent)
        if mutant == "no_depth_key":
            order = list(range(n))
        elif mutant == "ties_descending":
            order = sorted(range(n), key=lambda i: (int(dep[i]), -i))
        elif mutant == "depth_off_by_one_root":
            d2 = np.where(parent < 0, 2, dep)          # roots counted one too deep
            order = sorted(range(n), key=lambda i: (int(d2[i]), i))
        else:
            order = sorted(range(n), key=lambda i: (int(dep[i]), i))
        rank = np.empty(n, np.int64)
        for j, i in enumerate(order):
            rank[i] = j
        if mutant == "old_id_parents":
            parent_out = np.array([int(parent[i]) for i in order], np.int64)
        else:
            parent_out = np.array([-1 if parent[i] < 0 else int(rank[parent[i]]) for i in order], np.int64)
        return np.array(order, np.int64), rank, parent_out

    monkeypatch.setattr(R, "relabel_one", mutated)
    failed = False
    for check in (lambda: test_every_forest_under_random_labellings(4),
                  test_backwards_chain_comes_out_reversed, test_depth_sorted_tree_is_identity):
        try:
            check()
        except AssertionError:
            failed = True
    assert failed, f"mutant {mutant} survived every pin"

"""Pins for the top-w tree-construction oracle (oracle/grow.py).

The method is the modified DySpec best-first search of "Trees from Marginals"
(gist.science Technical Summary, Methodology, section 2 "Tree Construction"):
the top-w nodes of the candidate heap are expanded together.  Pins:
  * w = 1 is sequential best-first search: equal to a heapq-based search with
    the same draws (pop the best node, skip it at the depth cap, push children);
  * w >= N expands every frontier node each step: equal to a level-by-level
    construction (each level's nodes by score, then id);
  * invariants for any w: parents before children, depth <= max_depth,
    children score no higher than their parent, full trees while reachable;
  * planted mistakes (worst-first order, reversed ties, no depth cap, children
    assigned in id order, width off by one) must break one of the pins.
"""
import heapq

import numpy as np
import pytest

from oracle import grow as G
from gated_delta_net_gb300 import workloads as W


def _heap_best_first(cap, max_depth, c, e):
    f32 = np.float32
    parent, depth, score = [-1], [1], [f32(0.0)]
    heap = [(-0.0, 0)]
    while len(parent) < cap and heap:
        _, p = heapq.heappop(heap)
        if depth[p] >= max_depth:
            continue
        for j in range(int(min(c[p], e.shape[1]))):
            if len(parent) >= cap:
                break
            s = f32(score[p] - f32(e[p][j] * f32(j + 1)))
            parent.append(p)
            depth.append(depth[p] + 1)
            score.append(s)
            heapq.heappush(heap, (-float(s), len(parent) - 1))
    return parent, score


def _level_by_level(cap, max_depth, c, e):
    f32 = np.float32
    parent, depth, score = [-1], [1], [f32(0.0)]
    level = [0]
    while len(parent) < cap:
        level = [p for p in level if depth[p] < max_depth]
        if not level:
            break
        nxt = []
        for p in sorted(level, key=lambda i: (-float(score[i]), i)):
            for j in range(int(min(c[p], e.shape[1]))):
                if len(parent) >= cap:
                    break
                parent.append(p)
                depth.append(depth[p] + 1)
                score.append(f32(score[p] - f32(e[p][j] * f32(j + 1))))
                nxt.append(len(parent) - 1)
        level = nxt
    return parent, score


def _draws(seed, cap, maxc=8):
    return W.grow_draws(seed, np.array([0, cap]), maxc)


@pytest.mark.parametrize("seed,cap,depth", [(0, 128, 16), (1, 64, 4), (2, 200, 16), (3, 30, 2), (4, 256, 16)])
def test_width_one_is_heap_best_first(seed, cap, depth):
    c, e = _draws(seed, cap)
    par, sc, n = G.grow_one(cap, 1, depth, c, e)
    hp, hs = _heap_best_first(cap, depth, c, e)
    assert n == len(hp)
    assert list(par[:n]) == hp
    assert np.array_equal(sc[:n], np.array(hs, np.float32))


@pytest.mark.parametrize("seed,cap,depth", [(5, 128, 16), (6, 100, 5), (7, 256, 3)])
def test_unbounded_width_is_level_by_level(seed, cap, depth):
    c, e = _draws(seed, cap)
    par, sc, n = G.grow_one(cap, cap, depth, c, e)
    lp, ls = _level_by_level(cap, depth, c, e)
    assert list(par[:n]) == lp
    assert np.array_equal(sc[:n], np.array(ls, np.float32))


@pytest.mark.parametrize("width", [1, 2, 3, 8, 32])
def test_invariants(width):
    for seed in range(6):
        cap, D = 100, 16
        c, e = _draws(100 + seed, cap)
        par, sc, n = G.grow_one(cap, width, D, c, e)
        assert n == cap                      # geometric branching always fills 100 nodes at depth 16
        dep = np.zeros(n, int)
        for i in range(n):
            p = par[i]
            assert p < i
            dep[i] = 1 if p < 0 else dep[p] + 1
            if p >= 0:
                assert sc[i] <= sc[p]
        assert dep.max() <= D
        assert np.all(par[n:] == -1)


@pytest.mark.parametrize("width", [1, 3])
def test_ties_break_by_lower_id(width):
    # constant draws: cousins tie constantly (e.g. -1 - 1 = -2 = the root's second child)
    cap = 60
    c = np.full(cap, 2, np.int32)
    e = np.ones((cap, 8), np.float32)
    par, sc, n = G.grow_one(cap, width, 16, c, e)
    if width == 1:
        hp, hs = _heap_best_first(cap, 16, c, e)
        assert list(par[:n]) == hp
    # first steps by hand: the root, then its child 1 (score -1), then child 2 (-2)
    # ties with child 1's first child 3 (-2): the lower id, 2, goes first
    if width == 1:
        assert list(par[:7]) == [-1, 0, 0, 1, 1, 2, 2]
    else:
        # step 1 expands the root; step 2 expands nodes 1, 2 (the whole frontier)
        assert list(par[:7]) == [-1, 0, 0, 1, 1, 2, 2]
        # step 3: frontier 3 (-2), 4 (-3), 5 (-3), 6 (-4): ties 4, 5 -> 3, 4, 5 expanded
        assert list(par[7:13]) == [3, 3, 4, 4, 5, 5]


def test_depth_cap_can_end_a_tree_early():
    c = np.ones(50, np.int32)                # every expansion makes one child: a chain
    e = np.ones((50, 8), np.float32)
    par, sc, n = G.grow_one(50, 1, 5, c, e)
    assert n == 5 and list(par[:5]) == [-1, 0, 1, 2, 3]
    assert np.all(np.isneginf(sc[5:]))


@pytest.mark.parametrize("mutant", ["worst_first", "ties_reversed", "no_depth_cap", "children_by_id", "width_plus_one"])
def test_pins_catch_planted_mistakes(mutant, monkeypatch):
    real = G.grow_one

    def mutated(cap, width, max_depth, n_children, draws):
        f32 = np.float32
        parent, depth, score, expanded = [-1], [1], [f32(0.0)], [False]
        if mutant == "width_plus_one":
            width += 1
        while len(parent) < cap:
            frontier = [i for i in range(len(parent)) if not expanded[i] and
                        (mutant == "no_depth_cap" or depth[i] < max_depth)]
            if not frontier:
                break
            key = {"worst_first": lambda i: (float(score[i]), i),
                   "ties_reversed": lambda i: (-float(score[i]), -i)}.get(mutant, lambda i: (-float(score[i]), i))
            frontier.sort(key=key)
            chosen = frontier[:width]
            if mutant == "children_by_id":
                chosen = sorted(chosen)
            for p in chosen:
                expanded[p] = True
            for p in chosen:
                for j in range(int(min(n_children[p], draws.shape[1]))):
                    if len(parent) >= cap:
                        break
                    parent.append(p)
                    depth.append(depth[p] + 1)
                    score.append(f32(score[p] - f32(draws[p][j] * f32(j + 1))))
                    expanded.append(False)
        n = len(parent)
        par = np.full(cap, -1, np.int64)
        sc = np.full(cap, -np.inf, np.float32)
        par[:n], sc[:n] = parent, score
        return par, sc, n

    monkeypatch.setattr(G, "grow_one", mutated)
    failed = False
    checks = [lambda: test_width_one_is_heap_best_first(0, 128, 16),
              lambda: test_width_one_is_heap_best_first(3, 30, 2),
              lambda: test_unbounded_width_is_level_by_level(5, 128, 16),
              lambda: test_invariants(3), test_depth_cap_can_end_a_tree_early,
              lambda: test_ties_break_by_lower_id(1), lambda: test_ties_break_by_lower_id(3)]
    for check in checks:
        try:
            check()
        except AssertionError:
            failed = True
    assert failed, f"mutant {mutant} survived every pin"
    monkeypatch.setattr(G, "grow_one", real)

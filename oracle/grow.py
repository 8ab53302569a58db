"""Draft-tree construction by top-w best-first expansion: the plain CPU definition.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): the tests and the
benchmark's CPU-baseline leg call it; the CUDA library never does.

"Trees from Marginals" (gist.science Technical Summary, Methodology, section 2
"Tree Construction") builds the proposal tree with a modified DySpec
best-first search: instead of one expansion at a time, the top-w nodes are
taken from the candidate heap and expanded together (the wispaper.ai page,
"Dynamic Tree Construction", says the same).  The pages give no further
detail, so the reading taken here is:

  * node 0 is the root: score 0, depth 1; ids are given in creation order;
  * the frontier is every created node that is not yet expanded and whose
    depth is below max_depth;
  * one step takes the w best frontier nodes (score descending, then id
    ascending) and expands them in that order; expanding node p creates its
    c_p children j = 0 .. c_p - 1 with
        score = score_p - e_{p,j} * (j + 1)      (float32: multiply, then subtract)
    and depth_p + 1, until the request's capacity of N nodes is reached;
  * steps repeat until N nodes exist or the frontier is empty.

With w = 1 this is sequential best-first search; a larger w expands w nodes per
step, so a tree of N nodes takes about N / (w * mean children) steps instead of
N / mean children.  The random draws are inputs: c_p (children of node p if it
is expanded, at most max_children) and e_{p,j} >= 0, indexed by node id.
"""
from __future__ import annotations

import numpy as np


def grow_one(cap: int, width: int, max_depth: int, n_children, draws):
    """(parent, score, n) of one request; parent/score have `cap` entries, the
    rows at and past n are padding (parent -1, score -inf)."""
    f32 = np.float32
    parent, depth, score, expanded = [-1], [1], [f32(0.0)], [False]
    n_children = np.asarray(n_children)
    draws = np.asarray(draws, np.float32)
    maxc = draws.shape[1] if draws.ndim == 2 else 0
    while len(parent) < cap:
        frontier = [i for i in range(len(parent)) if not expanded[i] and depth[i] < max_depth]
        if not frontier:
            break
        frontier.sort(key=lambda i: (-float(score[i]), i))
        chosen = frontier[:width]
        for p in chosen:
            expanded[p] = True
        for p in chosen:
            c = int(min(max(int(n_children[p]), 0), maxc))
            for j in range(c):
                if len(parent) >= cap:
                    break
                parent.append(p)
                depth.append(depth[p] + 1)
                score.append(f32(score[p] - f32(draws[p][j] * f32(j + 1))))
                expanded.append(False)
    n = len(parent)
    par = np.full(cap, -1, np.int64)
    sc = np.full(cap, -np.inf, np.float32)
    par[:n] = parent
    sc[:n] = score
    return par, sc, n


def grow(node_offsets, width: int, max_depth: int, n_children, draws):
    """All requests (capacity = node_offsets[b+1] - node_offsets[b]): parent [T]
    (request-local), score [T] and n_nodes [B]."""
    T = int(node_offsets[-1])
    parent = np.full(T, -1, np.int64)
    score = np.full(T, -np.inf, np.float32)
    B = len(node_offsets) - 1
    n_nodes = np.zeros(B, np.int64)
    for b in range(B):
        lo, hi = int(node_offsets[b]), int(node_offsets[b + 1])
        if hi <= lo:
            continue
        p, s, n = grow_one(hi - lo, width, max_depth, n_children[lo:hi], draws[lo:hi])
        parent[lo:hi], score[lo:hi], n_nodes[b] = p, s, n
    return parent, score, n_nodes

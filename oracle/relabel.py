"""Topological relabelling of draft trees: the plain CPU definition.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): the tests and the
benchmark's CPU-baseline leg call it; the CUDA library never does.

"Trees from Marginals" (gist.science Technical Summary, section 3, Solution,
bullet 1) verifies a tree whose nodes are in topological order: every parent
comes before its children.  A tree handed over in any other order is relabelled
first.  The order used here is unique:

    nodes sorted by (depth, old id), depth = nodes on the root-to-node path.

A parent is one level shallower than its child, so it always sorts first.
Per request, for old ids i and new ids j:

    order[j] = the old id placed j-th,
    rank[i]  = the new id of old node i   (rank[order[j]] = j),
    parent_out[j] = rank[parent[order[j]]], or -1 for a root.

A request whose parent array is not a forest is malformed (status 1): a parent
outside [-1, n), a node that is its own parent, or a cycle.  Its outputs are
not defined.
"""
from __future__ import annotations

import numpy as np


def depths(parent: np.ndarray):
    """Depth of every node of one request (root = 1) by walking parent
    pointers; None if the array is not a forest."""
    n = len(parent)
    dep = np.zeros(n, np.int64)
    for i in range(n):
        # walk up until a node of known depth or a root; a walk longer than n
        # nodes has met a cycle
        chain = []
        j = i
        while j >= 0 and dep[j] == 0:
            p = int(parent[j])
            if p < -1 or p >= n or p == j or len(chain) > n:
                return None
            chain.append(j)
            j = p
        base = 0 if j < 0 else int(dep[j])
        for k, node in enumerate(reversed(chain)):
            dep[node] = base + k + 1
    return dep


def relabel_one(parent: np.ndarray):
    """(order, rank, parent_out) of one request, or None if malformed."""
    parent = np.asarray(parent, np.int64)
    dep = depths(parent)
    if dep is None:
        return None
    n = len(parent)
    order = sorted(range(n), key=lambda i: (int(dep[i]), i))
    rank = np.empty(n, np.int64)
    for j, i in enumerate(order):
        rank[i] = j
    parent_out = np.array([-1 if parent[i] < 0 else int(rank[parent[i]]) for i in order], np.int64)
    return np.array(order, np.int64), rank, parent_out


def relabel(parent: np.ndarray, node_offsets: np.ndarray):
    """All requests: (order, rank, parent_out, bad) with request-local ids;
    bad[b] is True for a malformed request (its rows are left at -1)."""
    parent = np.asarray(parent)
    T = len(parent)
    order = np.full(T, -1, np.int64)
    rank = np.full(T, -1, np.int64)
    parent_out = np.full(T, -1, np.int64)
    B = len(node_offsets) - 1
    bad = np.zeros(B, bool)
    for b in range(B):
        lo, hi = int(node_offsets[b]), int(node_offsets[b + 1])
        r = relabel_one(parent[lo:hi])
        if r is None:
            bad[b] = True
            continue
        order[lo:hi], rank[lo:hi], parent_out[lo:hi] = r
    return order, rank, parent_out, bad

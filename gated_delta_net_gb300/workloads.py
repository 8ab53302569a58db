"""Seeded synthetic inputs for speculative-tree verification through a GDN layer.

This module only draws inputs: tree shapes, token vectors, gates, the committed
state and the accepted path.  It holds none of the gated-delta-rule arithmetic,
so both the CUDA path and the float64 oracle can consume what it produces
without sharing any computation.

Shapes and distributions follow the workloads of *Trees from Marginals:
Autoregressive drafting with factorized priors* (Technical Summary, section 3
"Rollback-Free Tree Verification for GDN"; Experimental Results): a bf16
Qwen3.6-27B-like GDN layer with 16 key heads and 32 value heads of width 128,
proposal trees of up to a few hundred tokens and depth at most 16.

Value distributions (all workloads):
    q, k ~ N(0, 1), then L2-normalised per node and key head
    v    ~ N(0, 1)
    g    = -softplus(N(0, 1))          (log-decay, alpha = exp(g))
    beta = sigmoid(N(0, 1))
    S0   ~ N(0, 0.1^2)                 (layout [B, Hv, d_v, d_k])
For bf16 workloads q, k, v are rounded to bf16 (round to nearest even) here, so
both sides see bit-identical token values; g, beta and S0 stay float32.
"""
from __future__ import annotations

import dataclasses
import heapq
from typing import List, Optional, Sequence

import numpy as np

MAX_TREE_DEPTH = 16


@dataclasses.dataclass
class TreeBatch:
    """A batch of proposal trees plus every tensor one verify/commit call reads.

    Index conventions: node ids are request-local; ``parent[t] = -1`` marks a
    root (a child of the committed state S0); global row t of a request b is
    ``node_offsets[b] + local id``.  ``path_idx`` holds, per request, the local
    ids of the accepted root-to-leaf path (root first).
    """

    name: str
    batch: int
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    qkv_dtype: str                 # "f32" or "bf16"
    node_offsets: np.ndarray       # int32 [B+1]
    parent: np.ndarray             # int32 [T]
    q: np.ndarray                  # float32 [T, Hk, d_k] (bf16-exact when qkv_dtype == "bf16")
    k: np.ndarray                  # float32 [T, Hk, d_k]
    v: np.ndarray                  # float32 [T, Hv, d_v]
    g: np.ndarray                  # float32 [T, Hv]
    beta: np.ndarray               # float32 [T, Hv]
    S0: np.ndarray                 # float32 [B, Hv, d_v, d_k]
    path_offsets: np.ndarray       # int32 [B+1]
    path_idx: np.ndarray           # int32 [sum L]
    scale: float = 1.0
    max_depth_bound: int = 0       # declared bound on tree depth (0 = none declared)

    @property
    def total_nodes(self) -> int:
        return int(self.node_offsets[-1])

    @property
    def max_nodes(self) -> int:
        return int(np.max(np.diff(self.node_offsets))) if self.batch else 0

    def sizes(self) -> np.ndarray:
        return np.diff(self.node_offsets)


# ----------------------------------------------------------------------------
# value helpers (distribution only)
# ----------------------------------------------------------------------------

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _unit_rows(rng: np.random.Generator, shape) -> np.ndarray:
    x = rng.standard_normal(shape)
    x /= np.linalg.norm(x, axis=-1, keepdims=True)
    return x.astype(np.float32)


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


# ----------------------------------------------------------------------------
# tree shapes
# ----------------------------------------------------------------------------

def uniform_recursive_tree(rng: np.random.Generator, n: int) -> np.ndarray:
    """parent[0] = -1, parent[i] uniform over [0, i)."""
    parent = np.empty(n, dtype=np.int32)
    parent[0] = -1
    for i in range(1, n):
        parent[i] = rng.integers(0, i)
    return parent


def depth_capped_random_tree(rng: np.random.Generator, n: int,
                             max_depth: int = MAX_TREE_DEPTH) -> np.ndarray:
    """parent[i] uniform over {j < i : depth(j) < max_depth}; node 0 is the root."""
    parent = np.empty(n, dtype=np.int32)
    depth = np.empty(n, dtype=np.int32)
    parent[0] = -1
    depth[0] = 1
    open_nodes: List[int] = [0] if max_depth > 1 else []
    for i in range(1, n):
        p = open_nodes[rng.integers(0, len(open_nodes))]
        parent[i] = p
        depth[i] = depth[p] + 1
        if depth[i] < max_depth:
            open_nodes.append(i)
    return parent


def best_first_tree(rng: np.random.Generator, n: int,
                    max_depth: int = MAX_TREE_DEPTH) -> np.ndarray:
    """Best-first-like proposal tree.

    A max-heap is keyed on a synthetic log-score.  Each popped node below the
    depth cap gets c ~ Geometric(1/2) children (mean 2); child j of a node gets
    score = parent score - Exp(1) * (j + 1).  Ids are assigned in creation
    order, so every parent precedes its children.
    """
    parent = [-1]
    depth = [1]
    heap = [(-0.0, 0)]
    while len(parent) < n:
        if not heap:       # every frontier node sits at the cap: reopen a shallow node
            cands = [i for i in range(len(parent)) if depth[i] < max_depth]
            heap.append((-0.0, cands[rng.integers(0, len(cands))]))
        negscore, node = heapq.heappop(heap)
        if depth[node] >= max_depth:
            continue
        c = int(rng.geometric(0.5))
        for j in range(c):
            if len(parent) >= n:
                break
            cid = len(parent)
            parent.append(node)
            depth.append(depth[node] + 1)
            score = -negscore - rng.exponential(1.0) * (j + 1)
            heapq.heappush(heap, (-score, cid))
    return np.asarray(parent, dtype=np.int32)


def chainy_tree(rng: np.random.Generator, n: int, max_depth: int) -> np.ndarray:
    """Long paths: node i hangs under node i - 1 with probability 3/4 while that
    node is shallower than max_depth, else under a uniform node of depth
    < max_depth (node 0 is the root)."""
    parent = np.full(n, -1, dtype=np.int32)
    depth = np.ones(n, dtype=np.int32)
    for i in range(1, n):
        if depth[i - 1] < max_depth and rng.random() < 0.75:
            parent[i] = i - 1
        else:
            open_nodes = np.flatnonzero(depth[:i] < max_depth)
            parent[i] = int(rng.choice(open_nodes))
        depth[i] = depth[parent[i]] + 1
    return parent


def chain_tree(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def _walk_to_root(parent: np.ndarray, leaf: int) -> List[int]:
    path = []
    j = leaf
    while j >= 0:
        path.append(j)
        j = int(parent[j])
    return path[::-1]


def _path_lengths(parent: np.ndarray) -> np.ndarray:
    """Number of nodes on each root-to-node path (root = 1)."""
    n = len(parent)
    d = np.zeros(n, dtype=np.int32)
    for i in range(n):
        d[i] = 1 if parent[i] < 0 else d[parent[i]] + 1
    return d


def _leaves(parent: np.ndarray) -> np.ndarray:
    has_child = np.zeros(len(parent), dtype=bool)
    for p in parent:
        if p >= 0:
            has_child[p] = True
    return np.nonzero(~has_child)[0]


# ----------------------------------------------------------------------------
# accepted-path choices
# ----------------------------------------------------------------------------

def path_deepest_leaf(parent: np.ndarray, rng=None) -> List[int]:
    """Path to the deepest node (ties: lowest index)."""
    d = _path_lengths(parent)
    return _walk_to_root(parent, int(np.argmax(d)))


def path_whole_chain(parent: np.ndarray, rng=None) -> List[int]:
    return _walk_to_root(parent, len(parent) - 1)


def path_random_length(parent: np.ndarray, rng: np.random.Generator) -> List[int]:
    """Length L ~ U{1..16} clamped to the tree depth; end node uniform among depth-L nodes."""
    d = _path_lengths(parent)
    L = min(int(rng.integers(1, MAX_TREE_DEPTH + 1)), int(d.max()))
    cands = np.nonzero(d == L)[0]
    return _walk_to_root(parent, int(cands[rng.integers(0, len(cands))]))


def path_random_leaf(parent: np.ndarray, rng: np.random.Generator) -> List[int]:
    leaves = _leaves(parent)
    return _walk_to_root(parent, int(leaves[rng.integers(0, len(leaves))]))


# ----------------------------------------------------------------------------
# assembling a batch
# ----------------------------------------------------------------------------

def make_batch(name: str, seed: int, parents: Sequence[np.ndarray], n_k_heads: int,
               n_v_heads: int, d_k: int, d_v: int, qkv_dtype: str, path_fn,
               scale: float = 1.0, max_depth_bound: int = 0) -> TreeBatch:
    """Draw every tensor for the given tree shapes from one seeded PCG64 stream
    per request (``SeedSequence(seed).spawn``)."""
    B = len(parents)
    sizes = np.array([len(p) for p in parents], dtype=np.int64)
    offsets = np.zeros(B + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(sizes)
    T = int(offsets[-1])
    q = np.empty((T, n_k_heads, d_k), np.float32)
    k = np.empty((T, n_k_heads, d_k), np.float32)
    v = np.empty((T, n_v_heads, d_v), np.float32)
    g = np.empty((T, n_v_heads), np.float32)
    beta = np.empty((T, n_v_heads), np.float32)
    S0 = np.empty((B, n_v_heads, d_v, d_k), np.float32)
    paths = []
    children = np.random.SeedSequence(seed).spawn(B)
    for b in range(B):
        rng = np.random.Generator(np.random.PCG64(children[b]))
        lo, hi = offsets[b], offsets[b + 1]
        n = hi - lo
        q[lo:hi] = _unit_rows(rng, (n, n_k_heads, d_k))
        k[lo:hi] = _unit_rows(rng, (n, n_k_heads, d_k))
        v[lo:hi] = rng.standard_normal((n, n_v_heads, d_v)).astype(np.float32)
        g[lo:hi] = (-_softplus(rng.standard_normal((n, n_v_heads)))).astype(np.float32)
        beta[lo:hi] = _sigmoid(rng.standard_normal((n, n_v_heads))).astype(np.float32)
        S0[b] = (0.1 * rng.standard_normal((n_v_heads, d_v, d_k))).astype(np.float32)
        paths.append(path_fn(parents[b], rng) if n > 0 else [])
    if qkv_dtype == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    plens = np.array([len(p) for p in paths], dtype=np.int64)
    poff = np.zeros(B + 1, dtype=np.int32)
    poff[1:] = np.cumsum(plens)
    pidx = np.array([x for p in paths for x in p], dtype=np.int32)
    parent = (np.concatenate(parents).astype(np.int32) if B else np.zeros(0, np.int32))
    return TreeBatch(name, B, n_k_heads, n_v_heads, d_k, d_v, qkv_dtype, offsets, parent,
                     q, k, v, g, beta, S0, poff, pidx, scale, max_depth_bound)


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------

def tiny_tree(seed: int = 0) -> TreeBatch:
    """batch 1, one head, d_k = d_v = 16, N = 12, parent[i] uniform over [0, i), fp32;
    accepted path = the deepest leaf."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(2)[1]))
    parents = [uniform_recursive_tree(rng, 12)]
    return make_batch("tiny_tree", seed, parents, 1, 1, 16, 16, "f32", path_deepest_leaf)


def linear_chain(seed: int = 1) -> TreeBatch:
    """batch 1, 16 heads, d = 128, chain of N = 64 (parent[i] = i - 1), fp32;
    accepted path = the whole chain."""
    return make_batch("linear_chain", seed, [chain_tree(64)], 16, 16, 128, 128, "f32",
                      path_whole_chain)


def best_first(seed: int = 2, batch: int = 8, n: int = 128) -> TreeBatch:
    """batch 8, 16 key / 32 value heads, d = 128, N = 128 best-first-like trees of
    depth <= 16 with geometric(mean 2) branching; bf16 q/k/v; accepted-path
    length uniform in [1, 16]."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(batch + 1)[-1]))
    parents = [best_first_tree(rng, n) for _ in range(batch)]
    return make_batch("best_first", seed, parents, 16, 32, 128, 128, "bf16",
                      path_random_length, max_depth_bound=MAX_TREE_DEPTH)


def ragged_serving(seed: int = 3, batch: int = 64, n_lo: int = 16, n_hi: int = 128,
                   fixed_n: Optional[int] = None, name: str = "ragged_serving") -> TreeBatch:
    """batch 64, 16 key / 32 value heads, d = 128, per-request N uniform in [16, 128]
    (or fixed), random depth-capped trees (depth <= 16), bf16 q/k/v, fp32 state;
    accepted path = a uniformly chosen root-to-leaf path."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(batch + 1)[-1]))
    sizes = ([fixed_n] * batch if fixed_n is not None
             else [int(rng.integers(n_lo, n_hi + 1)) for _ in range(batch)])
    parents = [depth_capped_random_tree(rng, n) for n in sizes]
    return make_batch(name, seed, parents, 16, 32, 128, 128, "bf16", path_random_leaf,
                      max_depth_bound=MAX_TREE_DEPTH)


def serving_target(seed: int = 3, batch: int = 64, n: int = 128) -> TreeBatch:
    """The throughput point: batch 64, tree size 128 for every request, otherwise
    as ``ragged_serving``."""
    return ragged_serving(seed, batch, fixed_n=n, name=f"serving_b{batch}_n{n}")


def deep_serving(seed: int = 6, batch: int = 64, n: int = 128, max_depth: int = 32) -> TreeBatch:
    """Deep trees at the serving shapes: batch 64, tree size n, chain-like trees
    whose paths reach past 16 nodes (declared bound max_depth), 16 key / 32
    value heads, d = 128, bf16 q/k/v, fp32 state; accepted path = a uniformly
    chosen root-to-leaf path."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(batch + 1)[-1]))
    parents = [chainy_tree(rng, n, max_depth) for _ in range(batch)]
    return make_batch(f"deep_b{batch}_n{n}_d{max_depth}", seed, parents, 16, 32, 128, 128, "bf16",
                      path_random_leaf, max_depth_bound=max_depth)


SWEEP_N = (8, 16, 32, 64, 128, 256)
SWEEP_B = (1, 8, 32, 128)


def sweep_point(n: int, batch: int, seed: int = 4) -> TreeBatch:
    """One sweep point: fixed tree size n, the given batch, otherwise as ``ragged_serving``."""
    return ragged_serving(seed * 1000 + n * 7 + batch, batch, fixed_n=n,
                          name=f"sweep_b{batch}_n{n}")


def custom(seed: int, parents: Sequence[np.ndarray], n_k_heads: int = 1, n_v_heads: int = 1,
           d: int = 16, qkv_dtype: str = "f32", path_fn=path_random_leaf) -> TreeBatch:
    """Arbitrary shapes for edge-case tests."""
    return make_batch("custom", seed, parents, n_k_heads, n_v_heads, d, d, qkv_dtype, path_fn)


def grow_draws(seed: int, node_offsets: np.ndarray, max_children: int = 8):
    """Random inputs of the top-w tree construction, indexed by node row:
    children counts c ~ Geometric(1/2) clipped to [1, max_children] (mean about 2)
    and Exp(1) score decrements e [T][max_children], float32."""
    rng = np.random.default_rng(seed)
    T = int(node_offsets[-1])
    c = np.minimum(rng.geometric(0.5, T), max_children).astype(np.int32)
    e = rng.exponential(1.0, (T, max_children)).astype(np.float32)
    return c, e

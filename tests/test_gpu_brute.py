"""GPU against the oracle on every tree shape of six nodes (brute force).

"Trees from Marginals" (gist.science Technical Summary, section 3) verifies any
topologically ordered forest.  The oracle itself is pinned on the same
enumeration against numpy.linalg.solve of the matrix form
(tests/test_oracle_pins.py).  Here the CUDA path runs the whole enumeration:
  * every forest with parent[i] in [-1, i), N = 6 (720 shapes), in one launch;
  * the commit of every root-to-leaf path of every such forest.
Both the general kernels (fp32, d = 16) and the tensor-core kernels (bf16,
d = 128) are covered.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from gated_delta_net_gb300 import binding as gb
from gated_delta_net_gb300 import workloads as W

pytestmark = pytest.mark.gpu

N = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_net_gb300 import build
    build.build()
    gb.lib()


def _forests(n):
    return [np.array(f, np.int32) for f in itertools.product(*[range(-1, i) for i in range(n)])]


def _leaf_paths(parent):
    n = len(parent)
    has_child = np.zeros(n, bool)
    has_child[parent[parent >= 0]] = True
    paths = []
    for leaf in np.flatnonzero(~has_child):
        path, j = [], int(leaf)
        while j >= 0:
            path.append(j)
            j = int(parent[j])
        paths.append(path[::-1])
    return paths


def _rel(got, ref):
    return float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-30)


@pytest.mark.parametrize("dtype,d,tol", [("f32", 16, 1e-4), ("bf16", 128, 2e-2)])
def test_every_forest_verifies(dtype, d, tol):
    forests = _forests(N)
    assert len(forests) == 720
    tb = W.custom(600, forests, n_k_heads=1, n_v_heads=2, d=d, qkv_dtype=dtype)
    tb.max_depth_bound = N
    d_ = gb.upload(tb)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(d_["parent"], d_["node_offsets"], N, dev_status=status)
    o = gb.gdn_tree_verify(d_["q"], d_["k"], d_["v"], d_["g"], d_["beta"], d_["S0"], d_["node_offsets"],
                           d_["parent"], mask, depth, N, max_depth=N, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    assert _rel(o.float().cpu().numpy(), oracle.verify(tb)) <= tol


@pytest.mark.parametrize("dtype,d", [("f32", 16), ("bf16", 128)])
def test_every_leaf_path_of_every_forest_commits(dtype, d):
    reqs, paths = [], []
    for f in _forests(N):
        for path in _leaf_paths(f):
            reqs.append(f)
            paths.append(path)
    it = iter(paths)
    tb = W.custom(601, reqs, n_k_heads=1, n_v_heads=2, d=d, qkv_dtype=dtype,
                  path_fn=lambda p, r: next(it))
    d_ = gb.upload(tb)
    status = gb.new_status()
    S = gb.gdn_tree_commit(d_["k"], d_["v"], d_["g"], d_["beta"], d_["S0"], d_["node_offsets"],
                           d_["parent"], d_["path_offsets"], d_["path_idx"], N, max_path=N,
                           dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    ref, st = oracle.commit(tb)
    assert st == 0
    assert _rel(S.cpu().numpy(), ref) <= 1e-4

"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Tolerances: indices and masks bit-exact; fp32 inputs max|diff| <= 1e-4 * max|o|;
bf16 inputs max|diff| <= 2e-2 * max|o| (outputs are stored in the input dtype).
The committed state is fp32 and computed from the same (bf16-exact) inputs, so
it is held to 1e-4 * max|S| for every workload.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_net_gb300 import binding as gb
from gated_delta_net_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_F32, TOL_BF16, TOL_STATE = 1e-4, 2e-2, 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_net_gb300 import build
    build.build()
    gb.lib()


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = max(float(np.max(np.abs(ref))) if ref.size else 0.0, 1e-30)
    return float(np.max(np.abs(got - ref))) / scale if ref.size else 0.0


def tol_for(tb):
    return TOL_BF16 if tb.qkv_dtype == "bf16" else TOL_F32


def run_desc(d, tb, status):
    return gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], max(tb.max_nodes, 1),
                                  dev_status=status)


def run_verify(tb, impl="fused", out_dtype=None, d=None, max_depth=None):
    d = d or gb.upload(tb)
    status = gb.new_status()
    mask, depth = run_desc(d, tb, status)
    fn = gb.gdn_tree_verify if impl == "fused" else gb.gdn_tree_verify_branches
    o = fn(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
           mask, depth, max(tb.max_nodes, 1),
           max_depth=tb.max_depth_bound if max_depth is None else max_depth,
           scale=tb.scale, out_dtype=out_dtype, dev_status=status)
    torch.cuda.synchronize()
    return o, status, d


def run_commit(tb, d=None, inplace=False, max_path=0):
    d = d or gb.upload(tb)
    status = gb.new_status()
    out = d["S0"] if inplace else None
    S = gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                           d["parent"], d["path_offsets"], d["path_idx"], max(tb.max_nodes, 1),
                           max_path=max_path, out=out, dev_status=status)
    torch.cuda.synchronize()
    return S, status


NAMED = {
    "tiny_tree": lambda: W.tiny_tree(0),
    "linear_chain": lambda: W.linear_chain(1),
    "best_first": lambda: W.best_first(2),
    "ragged_serving": lambda: W.ragged_serving(3),
}


@pytest.fixture(scope="module")
def named():
    cache = {}

    def get(name):
        if name not in cache:
            tb = NAMED[name]()
            cache[name] = (tb, oracle.verify(tb), oracle.commit(tb)[0])
        return cache[name]
    return get


@pytest.mark.parametrize("name", list(NAMED))
def test_descriptor_bit_exact(name, named):
    tb, _, _ = named(name)
    d = gb.upload(tb)
    status = gb.new_status()
    mask, depth = run_desc(d, tb, status)
    words = mask.shape[1]
    ref_mask, ref_depth, st = oracle.build_desc(tb.parent, tb.node_offsets, words)
    assert st == 0 and int(status.item()) == 0
    np.testing.assert_array_equal(mask.cpu().numpy().view(np.uint32), ref_mask)
    np.testing.assert_array_equal(depth.cpu().numpy(), ref_depth)


@pytest.mark.parametrize("name", list(NAMED))
def test_verify_matches_oracle(name, named):
    tb, ref, _ = named(name)
    o, status, d = run_verify(tb)
    gb.check_status(status)
    assert rel_err(o.float().cpu().numpy(), ref) <= tol_for(tb)


@pytest.mark.parametrize("name", list(NAMED))
def test_branch_baseline_matches_oracle(name, named):
    tb, ref, _ = named(name)
    o, status, _ = run_verify(tb, impl="branches")
    gb.check_status(status)
    assert rel_err(o.float().cpu().numpy(), ref) <= tol_for(tb)


@pytest.mark.parametrize("name", list(NAMED))
def test_commit_matches_oracle(name, named):
    tb, _, ref = named(name)
    S, status = run_commit(tb)
    gb.check_status(status)
    assert rel_err(S.cpu().numpy(), ref) <= TOL_STATE


def test_commit_in_place(named):
    tb, _, ref = named("best_first")
    d = gb.upload(tb)
    S, status = run_commit(tb, d=d, inplace=True)
    gb.check_status(status)
    assert S.data_ptr() == d["S0"].data_ptr()
    assert rel_err(S.cpu().numpy(), ref) <= TOL_STATE


def test_verify_leaves_S0_untouched(named):
    tb, _, _ = named("best_first")
    d = gb.upload(tb)
    before = d["S0"].clone()
    run_verify(tb, d=d)
    assert torch.equal(before, d["S0"])


def test_fp32_output_from_bf16_inputs(named):
    tb, ref, _ = named("best_first")
    o, status, _ = run_verify(tb, out_dtype=torch.float32)
    gb.check_status(status)
    assert o.dtype == torch.float32
    assert rel_err(o.cpu().numpy(), ref) <= TOL_BF16


def test_verify_tree_sizes_sampled_against_oracle():
    """The throughput workload (batch 64, every tree 128 nodes) in the launch
    configuration the benchmark times, checked on sampled nodes."""
    tb = W.serving_target()
    o, status, _ = run_verify(tb)
    gb.check_status(status)
    rng = np.random.default_rng(0)
    sel = []
    for b in rng.choice(tb.batch, 16, replace=False):
        for h in rng.choice(tb.n_v_heads, 4, replace=False):
            for i in rng.choice(128, 8, replace=False):
                sel.append((b, h, i))
    ref = oracle.verify_selected(tb, sel)
    got = np.stack([o[tb.node_offsets[b] + i, h].float().cpu().numpy() for b, h, i in sel])
    assert rel_err(got, ref) <= TOL_BF16


def test_commit_full_throughput_workload():
    """The commit of the throughput workload (batch 64 x 32 value heads, every
    request's accepted path) in the benchmark's launch configuration, every state
    checked against the oracle."""
    tb = W.serving_target()
    S, status = run_commit(tb, max_path=tb.max_depth_bound)
    gb.check_status(status)
    ref, st = oracle.commit(tb)
    assert st == 0
    assert rel_err(S.cpu().numpy(), ref) <= TOL_STATE


def test_commit_verify_full_throughput_workload_sampled():
    """The serving-order call at full size: the previous tree's path committed,
    the next tree verified from the committed state; every committed state and
    sampled outputs checked against the oracle."""
    prev, new = W.serving_target(seed=41), W.serving_target(seed=42)
    dp, dn = gb.upload(prev), gb.upload(new)
    status = gb.new_status()
    mask, depth = run_desc(dn, new, status)
    o, S = gb.gdn_tree_commit_verify(dp, dp["S0"], prev.max_nodes, prev.max_depth_bound, dn["q"], dn["k"],
                                     dn["v"], dn["g"], dn["beta"], dn["node_offsets"], dn["parent"], mask,
                                     depth, new.max_nodes, max_depth=new.max_depth_bound, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    S_ref, st = oracle.commit(prev)
    assert st == 0
    assert rel_err(S.cpu().numpy(), S_ref) <= TOL_STATE
    new.S0 = S_ref
    rng = np.random.default_rng(1)
    sel = [(int(b), int(h), int(i)) for b in rng.choice(new.batch, 16, replace=False)
           for h in rng.choice(new.n_v_heads, 4, replace=False) for i in rng.choice(128, 8, replace=False)]
    ref = oracle.verify_selected(new, sel)
    got = np.stack([o[new.node_offsets[b] + i, h].float().cpu().numpy() for b, h, i in sel])
    assert rel_err(got, ref) <= TOL_BF16


@pytest.mark.parametrize("n,batch", [(8, 8), (16, 1), (32, 8), (64, 8), (128, 8), (256, 1),
                                     (256, 8)])
def test_sweep_points(n, batch):
    tb = W.sweep_point(n, batch)
    o, status, _ = run_verify(tb)
    gb.check_status(status)
    ob, status_b, _ = run_verify(tb, impl="branches")
    gb.check_status(status_b)
    rng = np.random.default_rng(n + batch)
    sel = [(int(rng.integers(batch)), int(rng.integers(tb.n_v_heads)), int(rng.integers(n)))
           for _ in range(96)]
    ref = oracle.verify_selected(tb, sel)
    for out in (o, ob):
        got = np.stack([out[tb.node_offsets[b] + i, h].float().cpu().numpy() for b, h, i in sel])
        assert rel_err(got, ref) <= TOL_BF16


# ----------------------------------------------------------------------------
# edge cases
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_head_dims_and_dtypes(d, dtype):
    rng = np.random.default_rng(d)
    parents = [W.uniform_recursive_tree(rng, n) for n in (1, 33, 7, 64)]
    tb = W.custom(d, parents, n_k_heads=2, n_v_heads=4, d=d, qkv_dtype=dtype)
    tb.scale = 0.5
    o, status, _ = run_verify(tb)
    gb.check_status(status)
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    assert rel_err(o.float().cpu().numpy(), oracle.verify(tb)) <= tol
    S, status = run_commit(tb)
    gb.check_status(status)
    assert rel_err(S.cpu().numpy(), oracle.commit(tb)[0]) <= TOL_STATE


def test_forest_and_empty_requests():
    rng = np.random.default_rng(1)
    forest = np.array([-1, -1, 0, 1, -1, 2, 3, 6, 4], np.int32)
    parents = [forest, np.zeros(0, np.int32), W.uniform_recursive_tree(rng, 31),
               np.zeros(0, np.int32), np.array([-1], np.int32)]
    tb = W.custom(5, parents, n_k_heads=1, n_v_heads=2, d=32)
    o, status, _ = run_verify(tb)
    gb.check_status(status)
    assert rel_err(o.cpu().numpy(), oracle.verify(tb)) <= TOL_F32
    S, status = run_commit(tb)
    gb.check_status(status)
    assert rel_err(S.cpu().numpy(), oracle.commit(tb)[0]) <= TOL_STATE


def test_max_size_chain_256():
    tb = W.custom(9, [W.chain_tree(256)], n_k_heads=1, n_v_heads=1, d=64,
                  path_fn=W.path_whole_chain)
    o, status, _ = run_verify(tb)
    gb.check_status(status)
    assert rel_err(o.cpu().numpy(), oracle.verify(tb)) <= TOL_F32
    S, status = run_commit(tb)
    gb.check_status(status)
    assert rel_err(S.cpu().numpy(), oracle.commit(tb)[0]) <= TOL_STATE


def test_empty_accepted_path_keeps_state():
    rng = np.random.default_rng(4)
    tb = W.custom(4, [W.uniform_recursive_tree(rng, 10)], d=16, path_fn=lambda p, r: [])
    S, status = run_commit(tb)
    gb.check_status(status)
    np.testing.assert_array_equal(S.cpu().numpy(), tb.S0)


def test_non_finite_inputs_stay_on_their_branch():
    """A NaN/Inf on one branch leaves every node outside its subtree bit-identical."""
    for dtype in ("f32", "bf16"):
        rng = np.random.default_rng(6)
        parent = W.depth_capped_random_tree(rng, 48, max_depth=8)
        tb = W.custom(6, [parent], n_k_heads=1, n_v_heads=2, d=128, qkv_dtype=dtype)
        base, st, _ = run_verify(tb)
        gb.check_status(st)
        bad_node = 5
        sub = {bad_node}
        for i in range(48):
            if parent[i] in sub:
                sub.add(i)
        for val in (np.nan, np.inf):
            tb2 = W.custom(6, [parent], n_k_heads=1, n_v_heads=2, d=128, qkv_dtype=dtype)
            tb2.k[bad_node] = val
            tb2.v[bad_node] = val
            tb2.g[bad_node] = val
            o2, st2, _ = run_verify(tb2)
            gb.check_status(st2)
            keep = [i for i in range(48) if i not in sub]
            assert torch.equal(o2[keep], base[keep])


def test_relabelled_tree_permutes_outputs():
    rng = np.random.default_rng(8)
    parent = W.depth_capped_random_tree(rng, 40, max_depth=6)
    children = {i: [] for i in range(40)}
    for i, p in enumerate(parent):
        if p >= 0:
            children[int(p)].append(i)
    order, frontier = [], [0]
    while frontier:
        order += frontier
        frontier = [c for f in frontier for c in reversed(children[f])]
    new_of = {old: new for new, old in enumerate(order)}
    perm = np.array(order)
    parent2 = np.array([new_of[int(parent[o])] if parent[o] >= 0 else -1 for o in order], np.int32)
    tb = W.custom(8, [parent], n_k_heads=1, n_v_heads=1, d=64)
    tb2 = W.custom(8, [parent2], n_k_heads=1, n_v_heads=1, d=64)
    tb2.q, tb2.k, tb2.v = tb.q[perm], tb.k[perm], tb.v[perm]
    tb2.g, tb2.beta, tb2.S0 = tb.g[perm], tb.beta[perm], tb.S0
    o, _, _ = run_verify(tb)
    o2, _, _ = run_verify(tb2)
    assert rel_err(o2.cpu().numpy(), o.cpu().numpy()[perm]) <= TOL_F32


# ----------------------------------------------------------------------------
# device-side error reporting
# ----------------------------------------------------------------------------

def test_bad_tree_sets_status():
    tb = W.custom(2, [np.array([-1, 0, 5, 1], np.int32)], d=16, path_fn=lambda p, r: [])
    o, status, _ = run_verify(tb)
    assert int(status.item()) & 1


def test_stale_descriptor_sets_status():
    tb = W.custom(2, [np.array([-1, 0, 1, 1], np.int32)], d=16)
    d = gb.upload(tb)
    status = gb.new_status()
    mask, depth = run_desc(d, tb, status)
    depth[3] = 7
    gb.gdn_tree_verify(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                       d["parent"], mask, depth, 4, dev_status=status)
    assert int(status.item()) & 32


def test_request_larger_than_max_nodes_sets_status():
    tb = W.custom(2, [W.chain_tree(40)], d=16)
    d = gb.upload(tb)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], 32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 4


@pytest.mark.parametrize("path", [[1], [0, 3], [0, 0], [0, 99], [0, 1, 3, 2]])
def test_bad_path_sets_status_and_leaves_state(path):
    parent = np.array([-1, 0, 0, 1], np.int32)
    tb = W.custom(3, [parent], d=16, path_fn=lambda p, r: path)
    d = gb.upload(tb)
    sentinel = torch.full_like(d["S0"], 7.0)
    status = gb.new_status()
    gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                       d["path_offsets"], d["path_idx"], 4, out=sentinel, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 2
    assert torch.all(sentinel == 7.0)


# ----------------------------------------------------------------------------
# the tcgen05 fast path (bf16, d = 128, <= 128 nodes, declared depth <= 16)
# ----------------------------------------------------------------------------

def _tc_batch(seed, sizes, hk=2, hv=4, max_depth=16, fn=None):
    rng = np.random.default_rng(seed)
    parents = [np.zeros(0, np.int32) if n == 0 else fn(rng, n) if fn
               else W.depth_capped_random_tree(rng, n, max_depth) for n in sizes]
    tb = W.custom(seed, parents, n_k_heads=hk, n_v_heads=hv, d=128, qkv_dtype="bf16")
    tb.max_depth_bound = 16
    return tb


@pytest.mark.parametrize("sizes", [(128,), (1, 2, 31, 32, 33), (100, 7, 128, 64, 65, 127),
                                   (5,) * 9])
def test_tc_path_sizes(sizes):
    tb = _tc_batch(sum(sizes), sizes)
    o, status, _ = run_verify(tb)
    gb.check_status(status)
    assert rel_err(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_tc_path_agrees_with_general_kernel():
    tb = _tc_batch(77, (128, 90, 128, 40))
    o_tc, st1, d = run_verify(tb)
    o_gen, st2, _ = run_verify(tb, d=d, max_depth=0)
    gb.check_status(st1)
    gb.check_status(st2)
    ref = oracle.verify(tb)
    e_tc = rel_err(o_tc.float().cpu().numpy(), ref)
    e_gen = rel_err(o_gen.float().cpu().numpy(), ref)
    assert e_tc <= TOL_BF16 and e_gen <= TOL_BF16


def test_tc_path_forest_and_chain16():
    forest = np.array([-1, 0, -1, 1, 2, -1, 3, 4, 6, 6], np.int32)
    tb = _tc_batch(3, (10, 16), fn=lambda r, n: forest if n == 10 else W.chain_tree(16))
    o, status, _ = run_verify(tb)
    gb.check_status(status)
    assert rel_err(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


@pytest.mark.parametrize("shape", ["star", "binary", "all_roots"])
def test_tc_path_tree_shapes(shape):
    # extreme shapes of 128 nodes: one root with 127 children (every descendant
    # row of the root full), a complete binary tree of depth 7, and 128 roots
    if shape == "star":
        par = np.array([-1] + [0] * 127, np.int32)
    elif shape == "binary":
        par = np.array([-1] + [(i - 1) // 2 for i in range(1, 127)], np.int32)
    else:
        par = np.full(128, -1, np.int32)
    tb = _tc_batch(61, (len(par), len(par)), fn=lambda r, n: par)
    o, status, _ = run_verify(tb)
    gb.check_status(status)
    assert rel_err(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_tc_path_fp32_output_and_scale():
    tb = _tc_batch(5, (128, 60))
    tb.scale = 0.25
    o, status, _ = run_verify(tb, out_dtype=torch.float32)
    gb.check_status(status)
    assert o.dtype == torch.float32
    assert rel_err(o.cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_tc_path_rejects_deeper_tree():
    tb = _tc_batch(4, (20, 30), fn=lambda r, n: W.chain_tree(n))
    o, status, _ = run_verify(tb)
    assert int(status.item()) & 8


def test_tc_path_non_finite_inputs_stay_on_their_branch():
    rng = np.random.default_rng(12)
    parent = W.depth_capped_random_tree(rng, 128, max_depth=10)
    base_tb = _tc_batch(12, (128,), hk=1, hv=2, fn=lambda r, n: parent)
    base, st, _ = run_verify(base_tb)
    gb.check_status(st)
    for bad_node in (0, 3, 77):
        sub = {bad_node}
        for i in range(128):
            if parent[i] in sub:
                sub.add(i)
        keep = [i for i in range(128) if i not in sub]
        for val in (np.nan, np.inf):
            tb2 = _tc_batch(12, (128,), hk=1, hv=2, fn=lambda r, n: parent)
            tb2.k[bad_node] = val
            tb2.v[bad_node] = val
            tb2.g[bad_node] = val
            o2, st2, _ = run_verify(tb2)
            gb.check_status(st2)
            assert torch.equal(o2[keep], base[keep])


def _mixed_sizes(count):
    cycle = (0, 1, 33, 128, 7, 64, 100, 2)
    return tuple(cycle[i % len(cycle)] for i in range(count))


def test_tc_path_many_items_per_block():
    # 240 requests x 4 value heads: more items than resident blocks, so each
    # persistent block runs several items of mixed sizes (and skips empty ones)
    tb = _tc_batch(21, _mixed_sizes(240))
    o, status, _ = run_verify(tb)
    gb.check_status(status)
    assert rel_err(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_tc_path_bad_request_among_many_is_skipped():
    tb = _tc_batch(22, _mixed_sizes(240))
    d = gb.upload(tb)
    status = gb.new_status()
    mask, depth = run_desc(d, tb, status)
    torch.cuda.synchronize()
    gb.check_status(status)
    bad = 11                                   # a request of 128 nodes
    lo, hi = int(tb.node_offsets[bad]), int(tb.node_offsets[bad + 1])
    depth[lo + 5] += 1                         # stale descriptor row
    out = torch.full((tb.total_nodes, tb.n_v_heads, tb.d_v), 5.0, dtype=torch.bfloat16,
                     device=d["q"].device)
    gb.gdn_tree_verify(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                       d["parent"], mask, depth, tb.max_nodes, max_depth=16, out=out,
                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 32
    assert torch.all(out[lo:hi] == 5.0)        # the malformed request is skipped
    ref = oracle.verify(tb)
    keep = np.r_[0:lo, hi:tb.total_nodes]
    assert rel_err(out.float().cpu().numpy()[keep], ref[keep]) <= TOL_BF16


def test_tc_path_leaves_S0_untouched():
    tb = _tc_batch(8, (128, 128))
    d = gb.upload(tb)
    before = d["S0"].clone()
    run_verify(tb, d=d)
    assert torch.equal(before, d["S0"])


# ----------------------------------------------------------------------------
# the TMA-staged commit (d = 128, declared path length <= 16)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["best_first", "ragged_serving"])
def test_fast_commit_matches_oracle(name, named):
    tb, _, ref = named(name)
    S, status = run_commit(tb, max_path=16)
    gb.check_status(status)
    assert rel_err(S.cpu().numpy(), ref) <= TOL_STATE


def test_fast_commit_in_place_and_target_workload():
    tb = W.serving_target(batch=16)
    d = gb.upload(tb)
    S, status = run_commit(tb, d=d, inplace=True, max_path=16)
    gb.check_status(status)
    assert S.data_ptr() == d["S0"].data_ptr()
    ref, st = oracle.commit(tb)
    assert st == 0
    assert rel_err(S.cpu().numpy(), ref) <= TOL_STATE


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fast_commit_edge_paths(dtype):
    rng = np.random.default_rng(31)
    parents = [W.depth_capped_random_tree(rng, n, 16) for n in (1, 5, 40, 128)] + [W.chain_tree(16)]
    for fn in (W.path_random_leaf, lambda p, r: [], W.path_deepest_leaf):
        tb = W.custom(31, parents, n_k_heads=2, n_v_heads=4, d=128, qkv_dtype=dtype, path_fn=fn)
        S, status = run_commit(tb, max_path=16)
        gb.check_status(status)
        assert rel_err(S.cpu().numpy(), oracle.commit(tb)[0]) <= TOL_STATE


def test_fast_commit_flags_long_and_bad_paths():
    tb = W.custom(2, [W.chain_tree(20)], d=128, path_fn=W.path_whole_chain)
    d = gb.upload(tb)
    sentinel = torch.full_like(d["S0"], 3.0)
    status = gb.new_status()
    gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                       d["path_offsets"], d["path_idx"], 20, max_path=16, out=sentinel,
                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 8
    assert torch.all(sentinel == 3.0)
    parent = np.array([-1, 0, 0, 1], np.int32)
    tb = W.custom(3, [parent], d=128, path_fn=lambda p, r: [0, 3])
    d = gb.upload(tb)
    sentinel = torch.full_like(d["S0"], 3.0)
    status = gb.new_status()
    gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                       d["path_offsets"], d["path_idx"], 4, max_path=16, out=sentinel,
                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 2
    assert torch.all(sentinel == 3.0)


def test_fast_commit_many_items_with_a_bad_path():
    # more items than resident blocks, mixed sizes and empty requests; one
    # request's path is reversed (not root-first): it alone is flagged and skipped
    tb = _tc_batch(23, _mixed_sizes(240))
    lens = np.diff(tb.path_offsets)
    bad = int(np.flatnonzero(lens >= 2)[3])
    a, e = int(tb.path_offsets[bad]), int(tb.path_offsets[bad + 1])
    tb.path_idx[a:e] = tb.path_idx[a:e][::-1].copy()
    d = gb.upload(tb)
    sentinel = torch.full_like(d["S0"], 3.0)
    status = gb.new_status()
    gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                       d["path_offsets"], d["path_idx"], tb.max_nodes, max_path=16, out=sentinel,
                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2
    assert torch.all(sentinel[bad] == 3.0)
    ref, st = oracle.commit(tb)
    assert st == 2
    keep = [r for r in range(tb.batch) if r != bad]
    assert rel_err(sentinel.cpu().numpy()[keep], ref[keep]) <= TOL_STATE

"""GPU parity of gdn_tree_commit_verify: the delayed commit of the previous
tree's accepted path followed by the verification of the next tree from the
committed state, the verification launched as the commit's programmatic
dependent ("Trees from Marginals", gist.science Technical Summary, section 3,
Solution, bullet 4: the state is committed in the next decoding iteration).

Reference: oracle.commit on the previous tree (the committed state, fp32
tolerance 1e-4 * max|S|), then oracle.verify of the new tree from that state
(bf16 tolerance 2e-2 * max|o|; fp32 1e-4 relative).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_net_gb300 import binding as gb
from gated_delta_net_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_STATE, TOL_BF16 = 1e-4, 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_net_gb300 import build
    build.build()
    gb.lib()


def _rel(got, ref):
    return float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-30)


def _run(prev, new, in_place=False, S_new_init=None):
    dp, dn = gb.upload(prev), gb.upload(new)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(dn["parent"], dn["node_offsets"], new.max_nodes, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    S0 = dp["S0"]
    S_new = S0 if in_place else (S_new_init if S_new_init is not None else torch.empty_like(S0))
    S0_before = S0.clone()
    o, S = gb.gdn_tree_commit_verify(dp, S0, prev.max_nodes, 16, dn["q"], dn["k"], dn["v"], dn["g"],
                                     dn["beta"], dn["node_offsets"], dn["parent"], mask, depth,
                                     new.max_nodes, max_depth=16, S_new=S_new, dev_status=status)
    torch.cuda.synchronize()
    return o, S, status, S0_before


def _reference(prev, new):
    S_ref, st = oracle.commit(prev)
    assert st == 0
    new.S0 = S_ref                 # the new tree is verified from the committed state
    return S_ref, oracle.verify(new)


def test_commit_then_verify_matches_the_oracle():
    prev, new = W.serving_target(seed=21, batch=6), W.serving_target(seed=22, batch=6)
    o, S, status, _ = _run(prev, new)
    gb.check_status(status)
    S_ref, o_ref = _reference(prev, new)
    assert _rel(S.cpu().numpy(), S_ref) <= TOL_STATE
    assert _rel(o.float().cpu().numpy(), o_ref) <= TOL_BF16


def test_in_place_and_ragged_many_items():
    # 80 requests x 32 value heads: several items per persistent block; ragged
    # trees on both sides; the state committed in place
    prev = W.ragged_serving(seed=23, batch=80)
    new = W.ragged_serving(seed=24, batch=80)
    o, S, status, S0_before = _run(prev, new, in_place=True)
    gb.check_status(status)
    prev.S0 = S0_before.cpu().numpy()
    S_ref, o_ref = _reference(prev, new)
    assert _rel(S.cpu().numpy(), S_ref) <= TOL_STATE
    assert _rel(o.float().cpu().numpy(), o_ref) <= TOL_BF16


def test_empty_previous_path_keeps_the_state_exactly():
    parents = [W.depth_capped_random_tree(np.random.default_rng(s), 40, 16) for s in range(3)]
    prev = W.custom(25, parents, n_k_heads=2, n_v_heads=4, d=128, qkv_dtype="bf16", path_fn=lambda p, r: [])
    new = W.custom(26, parents, n_k_heads=2, n_v_heads=4, d=128, qkv_dtype="bf16")
    o, S, status, S0_before = _run(prev, new)
    gb.check_status(status)
    assert torch.equal(S, S0_before)
    new.S0 = S0_before.cpu().numpy().astype(np.float64)
    assert _rel(o.float().cpu().numpy(), oracle.verify(new)) <= TOL_BF16


def test_general_shapes_chain_the_general_kernels():
    # fp32 tokens, d = 16, a deep chain: neither tensor-core kernel applies
    parents = [np.arange(-1, 39, dtype=np.int32), W.depth_capped_random_tree(np.random.default_rng(5), 30, 40)]
    prev = W.custom(29, parents, n_k_heads=2, n_v_heads=4, d=16, qkv_dtype="f32")
    new = W.custom(30, parents, n_k_heads=2, n_v_heads=4, d=16, qkv_dtype="f32")
    dp, dn = gb.upload(prev), gb.upload(new)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(dn["parent"], dn["node_offsets"], new.max_nodes, dev_status=status)
    o, S = gb.gdn_tree_commit_verify(dp, dp["S0"], prev.max_nodes, 0, dn["q"], dn["k"], dn["v"], dn["g"],
                                     dn["beta"], dn["node_offsets"], dn["parent"], mask, depth,
                                     new.max_nodes, max_depth=0, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    S_ref, o_ref = _reference(prev, new)
    assert _rel(S.cpu().numpy(), S_ref) <= TOL_STATE
    assert _rel(o.float().cpu().numpy(), o_ref) <= TOL_STATE


def test_tensor_core_verify_after_the_general_commit():
    # max_path = 0 (unknown) sends the commit to the general kernel, which never
    # signals its dependents early; the tensor-core verify is still launched as its
    # programmatic dependent and must still see the whole committed state
    prev, new = W.serving_target(seed=33, batch=5), W.serving_target(seed=34, batch=5)
    dp, dn = gb.upload(prev), gb.upload(new)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(dn["parent"], dn["node_offsets"], new.max_nodes, dev_status=status)
    o, S = gb.gdn_tree_commit_verify(dp, dp["S0"], prev.max_nodes, 0, dn["q"], dn["k"], dn["v"], dn["g"],
                                     dn["beta"], dn["node_offsets"], dn["parent"], mask, depth,
                                     new.max_nodes, max_depth=16, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    S_ref, o_ref = _reference(prev, new)
    assert _rel(S.cpu().numpy(), S_ref) <= TOL_STATE
    assert _rel(o.float().cpu().numpy(), o_ref) <= TOL_BF16


def test_replays_in_a_cuda_graph():
    prev, new = W.serving_target(seed=31, batch=4), W.serving_target(seed=32, batch=4)
    dp, dn = gb.upload(prev), gb.upload(new)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(dn["parent"], dn["node_offsets"], new.max_nodes, dev_status=status)
    S_new = torch.empty_like(dp["S0"])
    o = torch.empty((new.total_nodes, new.n_v_heads, new.d_v), dtype=torch.bfloat16, device="cuda")

    def call():
        gb.gdn_tree_commit_verify(dp, dp["S0"], prev.max_nodes, 16, dn["q"], dn["k"], dn["v"], dn["g"],
                                  dn["beta"], dn["node_offsets"], dn["parent"], mask, depth, new.max_nodes,
                                  S_new=S_new, out=o, dev_status=status, stream=torch.cuda.current_stream())

    call()
    torch.cuda.synchronize()
    gb.check_status(status)
    o_eager, S_eager = o.clone(), S_new.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(3):
        o.zero_()
        S_new.zero_()
        graph.replay()
        torch.cuda.synchronize()
        gb.check_status(status)
        assert torch.equal(o, o_eager) and torch.equal(S_new, S_eager)


def test_bad_previous_path_is_flagged_and_left_unwritten():
    parent = W.depth_capped_random_tree(np.random.default_rng(3), 30, 16)
    parents = [parent, parent, parent]
    assert parent[0] == -1 and parent[1] == 0
    paths = iter([[0, 1], [1], [0]])            # the second is not root-first
    prev = W.custom(27, parents, n_k_heads=1, n_v_heads=2, d=128, qkv_dtype="bf16",
                    path_fn=lambda p, r: next(paths))
    new = W.custom(28, parents, n_k_heads=1, n_v_heads=2, d=128, qkv_dtype="bf16")
    sentinel = torch.full((3, 2, 128, 128), 3.0, device="cuda")
    dn = gb.upload(new)
    o_init = torch.full((new.total_nodes, 2, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    dp = gb.upload(prev)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(dn["parent"], dn["node_offsets"], 30, dev_status=status)
    gb.gdn_tree_commit_verify(dp, dp["S0"], 30, 16, dn["q"], dn["k"], dn["v"], dn["g"], dn["beta"],
                              dn["node_offsets"], dn["parent"], mask, depth, 30, S_new=sentinel,
                              out=o_init, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2                   # GDN_DEV_BAD_PATH
    assert torch.all(sentinel[1] == 3.0)             # the bad request's state is not committed
    assert not torch.all(sentinel[0] == 3.0) and not torch.all(sentinel[2] == 3.0)
    assert not torch.all(o_init[:30] == 5.0)


# ----------------------------------------------------------------------------
# edge cases of the chained call on the tensor-core kernels (bf16, d = 128,
# max_path <= 16, new trees of at most 128 nodes with depth <= 16)
# ----------------------------------------------------------------------------

DEV_BAD_PATH, DEV_TOO_DEEP, DEV_TIMEOUT = 2, 8, 16


def _trees(seed, sizes):
    rng = np.random.default_rng(seed)
    return [W.depth_capped_random_tree(rng, n, 16) if n > 0 else np.zeros(0, np.int32) for n in sizes]


def test_odd_value_head_groups_in_place():
    # 6 value heads over 2 key heads: the verification's second pair of each key
    # head holds one head
    prev = W.custom(41, _trees(40, [50, 70, 90]), n_k_heads=2, n_v_heads=6, d=128, qkv_dtype="bf16")
    new = W.custom(42, _trees(43, [90, 30, 128]), n_k_heads=2, n_v_heads=6, d=128, qkv_dtype="bf16")
    o, S, status, S0_before = _run(prev, new, in_place=True)
    gb.check_status(status)
    prev.S0 = S0_before.cpu().numpy()
    S_ref, o_ref = _reference(prev, new)
    assert _rel(S.cpu().numpy(), S_ref) <= TOL_STATE
    assert _rel(o.float().cpu().numpy(), o_ref) <= TOL_BF16


@pytest.mark.parametrize("batch", [6, 320])
def test_requests_with_empty_new_trees_are_still_committed(batch):
    # every third new tree is empty: those requests verify nothing but are still
    # committed (batch 320: more verification units than SMs)
    rng = np.random.default_rng(50 + batch)
    prev_sizes = [int(rng.integers(2, 24)) for _ in range(batch)]
    new_sizes = [0 if r % 3 == 1 else int(rng.integers(1, 24)) for r in range(batch)]
    prev = W.custom(51, _trees(52, prev_sizes), n_k_heads=1, n_v_heads=2, d=128, qkv_dtype="bf16")
    new = W.custom(53, _trees(54, new_sizes), n_k_heads=1, n_v_heads=2, d=128, qkv_dtype="bf16",
                   path_fn=lambda p, r: [])
    o, S, status, _ = _run(prev, new)
    gb.check_status(status)
    S_ref, o_ref = _reference(prev, new)
    assert _rel(S.cpu().numpy(), S_ref) <= TOL_STATE
    assert _rel(o.float().cpu().numpy(), o_ref) <= TOL_BF16


def test_path_past_max_path_is_flagged_and_left_unwritten():
    # request 0 accepts a 20-node chain against max_path = 16
    chain = np.arange(-1, 19, dtype=np.int32)
    tree = _trees(60, [40])[0]
    leaf_path = W.path_random_leaf(tree, np.random.default_rng(61))
    paths = iter([list(range(20)), leaf_path])
    prev = W.custom(62, [chain, tree], n_k_heads=1, n_v_heads=2, d=128, qkv_dtype="bf16",
                    path_fn=lambda p, r: next(paths))
    new = W.custom(63, [tree, tree], n_k_heads=1, n_v_heads=2, d=128, qkv_dtype="bf16")
    sentinel = torch.full((2, 2, 128, 128), 3.0, device="cuda")
    o, S, status, _ = _run(prev, new, S_new_init=sentinel)
    assert int(status.item()) == DEV_TOO_DEEP
    assert torch.all(S[0] == 3.0)
    S_ref, st = oracle.commit(prev)      # the oracle has no path bound
    assert st == 0
    assert _rel(S[1].cpu().numpy(), S_ref[1]) <= TOL_STATE
    new.S0 = S_ref
    o_ref = oracle.verify(new)
    lo = int(new.node_offsets[1])
    assert _rel(o[lo:].float().cpu().numpy(), o_ref[lo:]) <= TOL_BF16


def test_fp32_outputs():
    prev, new = W.serving_target(seed=71, batch=3), W.serving_target(seed=72, batch=3)
    dp, dn = gb.upload(prev), gb.upload(new)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(dn["parent"], dn["node_offsets"], new.max_nodes, dev_status=status)
    o, S = gb.gdn_tree_commit_verify(dp, dp["S0"], prev.max_nodes, 16, dn["q"], dn["k"], dn["v"], dn["g"],
                                     dn["beta"], dn["node_offsets"], dn["parent"], mask, depth,
                                     new.max_nodes, max_depth=16, out_dtype=torch.float32, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    assert o.dtype == torch.float32
    S_ref, o_ref = _reference(prev, new)
    assert _rel(S.cpu().numpy(), S_ref) <= TOL_STATE
    assert _rel(o.cpu().numpy(), o_ref) <= TOL_BF16


def test_wait_probe_times_out_and_the_chained_kernels_return():
    prev, new = W.serving_target(seed=81, batch=3), W.serving_target(seed=82, batch=3)
    o0, S0, status, _ = _run(prev, new)
    gb.check_status(status)
    try:
        gb.gdn_test_set_wait_probe(2000)
        o1, S1, status1, _ = _run(prev, new)
        bits = int(status1.item())
    finally:
        gb.gdn_test_set_wait_probe(0)
    assert bits == DEV_TIMEOUT
    assert torch.equal(o1, o0) and torch.equal(S1, S0)
    o2, S2, status2, _ = _run(prev, new)
    gb.check_status(status2)
    assert torch.equal(o2, o0) and torch.equal(S2, S0)

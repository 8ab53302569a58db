"""GPU parity of the tensor-core verify for trees of 129 to 256 nodes (bf16,
d = 128, depth <= 16): two node tiles per request, block-lower-triangular P.

Every case compares with the float64 oracle ("Trees from Marginals",
gist.science Technical Summary, section 3 "Rollback-Free Tree Verification
for GDN") at the bf16 bar, max|diff| <= 2e-2 * max|o|; batches mix requests of
at most 128 nodes (one tile) with wider ones, since a batch whose largest tree
has more than 128 nodes runs every request on this kernel.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_net_gb300 import binding as gb
from gated_delta_net_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
DEV_TOO_DEEP, DEV_BAD_DESC = 8, 32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_net_gb300 import build
    build.build()
    gb.lib()


def _rel(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-30)


def _batch(seed, sizes, hk=2, hv=4, fn=None):
    rng = np.random.default_rng(seed)
    parents = [np.zeros(0, np.int32) if n == 0 else fn(rng, n) if fn
               else W.depth_capped_random_tree(rng, n, 16) for n in sizes]
    tb = W.custom(seed, parents, n_k_heads=hk, n_v_heads=hv, d=128, qkv_dtype="bf16")
    tb.max_depth_bound = 16
    return tb


def _verify(tb, d=None, max_depth=16, out=None, out_dtype=None, words=None):
    d = d or gb.upload(tb)
    status = gb.new_status()
    kw = {} if words is None else {"mask_words": words}
    mask, depth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes,
                                         dev_status=status, **kw)
    o = gb.gdn_tree_verify(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                           d["parent"], mask, depth, tb.max_nodes, max_depth=max_depth,
                           scale=tb.scale, out=out, out_dtype=out_dtype, dev_status=status)
    torch.cuda.synchronize()
    return o, status, d


@pytest.mark.parametrize("sizes", [(256,), (129,), (200, 1, 128, 0, 255, 130, 64),
                                   (160, 33, 31, 32, 256)])
def test_wide_sizes(sizes):
    tb = _batch(sum(sizes) + 3, sizes)
    o, status, _ = _verify(tb)
    gb.check_status(status)
    assert _rel(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_wide_agrees_with_general_kernel():
    tb = _batch(81, (256, 140, 7, 222))
    o_w, st1, d = _verify(tb)
    o_gen, st2, _ = _verify(tb, d=d, max_depth=0)
    gb.check_status(st1)
    gb.check_status(st2)
    ref = oracle.verify(tb)
    assert _rel(o_w.float().cpu().numpy(), ref) <= TOL_BF16
    assert _rel(o_gen.float().cpu().numpy(), ref) <= TOL_BF16


@pytest.mark.parametrize("shape", ["star", "binary", "all_roots", "chains"])
def test_wide_tree_shapes(shape):
    # a root with 255 children (its descendant row spans all eight words), a
    # complete binary tree of 255 nodes (depth 8, ancestors across both tiles),
    # 256 roots, and sixteen chains of 16 whose later chains sit in the second tile
    if shape == "star":
        par = np.array([-1] + [0] * 255, np.int32)
    elif shape == "binary":
        par = np.array([-1] + [(i - 1) // 2 for i in range(1, 255)], np.int32)
    elif shape == "all_roots":
        par = np.full(256, -1, np.int32)
    else:
        par = np.array([-1 if i % 16 == 0 else i - 1 for i in range(256)], np.int32)
    tb = _batch(62, (len(par), len(par), 90), fn=lambda r, n: par if n == len(par) else
                W.depth_capped_random_tree(r, n, 16))
    o, status, _ = _verify(tb)
    gb.check_status(status)
    assert _rel(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_wide_chain16_across_the_tile_boundary():
    # one chain of 16 from node 120 to node 135 under a root chain: the path of a
    # second-tile node runs through first-tile ancestors (the P21 block)
    par = np.array([-1] + list(range(0, 119)) + [-1] + list(range(120, 135)) +
                   [-1] * 120, np.int32)
    par[1:120] = np.where(np.arange(1, 120) % 15 == 0, -1, par[1:120])
    tb = _batch(63, (len(par),), hk=1, hv=2, fn=lambda r, n: par)
    depth = np.zeros(len(par), np.int64)
    for i, a in enumerate(par):
        depth[i] = 1 if a < 0 else depth[a] + 1
    assert depth.max() == 16 and depth[135] == 16
    o, status, _ = _verify(tb)
    gb.check_status(status)
    assert _rel(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_wide_fp32_output_and_scale():
    tb = _batch(64, (256, 150))
    tb.scale = 0.25
    o, status, _ = _verify(tb, out_dtype=torch.float32)
    gb.check_status(status)
    assert o.dtype == torch.float32
    assert _rel(o.cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_wide_rejects_deeper_tree():
    tb = _batch(65, (200, 30), fn=lambda r, n: W.chain_tree(n))
    _, status, _ = _verify(tb)
    assert int(status.item()) & DEV_TOO_DEEP


def test_wide_non_finite_inputs_stay_on_their_branch():
    rng = np.random.default_rng(13)
    parent = W.depth_capped_random_tree(rng, 256, max_depth=12)
    base_tb = _batch(13, (256,), hk=1, hv=2, fn=lambda r, n: parent)
    base, st, _ = _verify(base_tb)
    gb.check_status(st)
    for bad_node in (0, 5, 127, 128, 201):
        sub = {bad_node}
        for i in range(256):
            if parent[i] in sub:
                sub.add(i)
        keep = [i for i in range(256) if i not in sub]
        for val in (np.nan, np.inf):
            tb2 = _batch(13, (256,), hk=1, hv=2, fn=lambda r, n: parent)
            tb2.k[bad_node] = val
            tb2.v[bad_node] = val
            tb2.g[bad_node] = val
            o2, st2, _ = _verify(tb2)
            gb.check_status(st2)
            assert torch.equal(o2[keep], base[keep])


def _mixed_sizes(count):
    cycle = (0, 1, 33, 256, 7, 129, 200, 2, 128)
    return tuple(cycle[i % len(cycle)] for i in range(count))


def test_wide_many_items_per_block():
    # 180 requests x 4 value heads: more items than resident blocks, so each
    # persistent block runs several items of mixed sizes (and skips empty ones)
    tb = _batch(23, _mixed_sizes(180))
    o, status, _ = _verify(tb)
    gb.check_status(status)
    assert _rel(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_wide_bad_request_among_many_is_skipped():
    tb = _batch(24, _mixed_sizes(180))
    d = gb.upload(tb)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes,
                                         dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    bad = 15                                   # a request of 200 nodes
    lo, hi = int(tb.node_offsets[bad]), int(tb.node_offsets[bad + 1])
    assert hi - lo == 200
    depth[lo + 170] += 1                       # stale descriptor row in the second tile
    out = torch.full((tb.total_nodes, tb.n_v_heads, tb.d_v), 5.0, dtype=torch.bfloat16,
                     device=d["q"].device)
    gb.gdn_tree_verify(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                       d["parent"], mask, depth, tb.max_nodes, max_depth=16, out=out,
                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == DEV_BAD_DESC
    assert torch.all(out[lo:hi] == 5.0)        # the malformed request is skipped
    ref = oracle.verify(tb)
    keep = np.r_[0:lo, hi:tb.total_nodes]
    assert _rel(out.float().cpu().numpy()[keep], ref[keep]) <= TOL_BF16


def test_wide_stray_bit_past_the_tree_is_a_stale_descriptor():
    # descriptor rows of eight words for trees of at most 180 nodes: the words
    # past the tree are read and must be empty
    tb = _batch(25, (180, 97, 150))
    o6, status6, d = _verify(tb)
    gb.check_status(status6)
    o, status, _ = _verify(tb, d=d, words=8)
    gb.check_status(status)
    assert torch.equal(o, o6)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes,
                                         mask_words=8, dev_status=status)
    torch.cuda.synchronize()
    mask[5, 7] = 1                             # request 0, node 5: a bit for node 224
    out = torch.full((tb.total_nodes, tb.n_v_heads, tb.d_v), 3.0, dtype=torch.bfloat16,
                     device=d["q"].device)
    gb.gdn_tree_verify(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                       d["parent"], mask, depth, tb.max_nodes, max_depth=16, out=out,
                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == DEV_BAD_DESC
    assert torch.all(out[:180] == 3.0)         # the request is skipped
    assert torch.equal(out[180:], o6[180:])


def test_wide_leaves_S0_untouched():
    tb = _batch(26, (256, 256))
    d = gb.upload(tb)
    before = d["S0"].clone()
    _verify(tb, d=d)
    assert torch.equal(before, d["S0"])


def test_wide_wait_probe_times_out_and_returns():
    tb = _batch(27, (256, 133, 256))
    o0, st, d = _verify(tb)
    gb.check_status(st)
    try:
        gb.gdn_test_set_wait_probe(2000)
        o1, st1, _ = _verify(tb, d=d)
        bits = int(st1.item())
    finally:
        gb.gdn_test_set_wait_probe(0)
    assert bits == 16
    assert torch.equal(o1, o0)
    o2, st2, _ = _verify(tb, d=d)
    gb.check_status(st2)
    assert torch.equal(o2, o0)


def test_wide_commit_verify_serving_order():
    # the committed state of the previous tree feeds the verify of the next one,
    # the verify launched as the commit's programmatic dependent
    prev = _batch(28, (256, 180))
    new = _batch(29, (256, 200))
    dp, dn = gb.upload(prev), gb.upload(new)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(dn["parent"], dn["node_offsets"], new.max_nodes,
                                         dev_status=status)
    o, S = gb.gdn_tree_commit_verify(dp, dp["S0"], prev.max_nodes, 16, dn["q"], dn["k"], dn["v"],
                                     dn["g"], dn["beta"], dn["node_offsets"], dn["parent"], mask,
                                     depth, new.max_nodes, max_depth=16, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    S_ref, st = oracle.commit(prev)
    assert st == 0
    new.S0 = S_ref.astype(np.float32)
    assert _rel(o.float().cpu().numpy(), oracle.verify(new)) <= TOL_BF16


# ----------------------------------------------------------------------------
# one tile, paths of 17 to 32 nodes (declared max_depth 17..32, N <= 128)
# ----------------------------------------------------------------------------

def _deep_tree(rng, n, cap):
    """Mostly chain-like: node i hangs under node i - 1 with probability 3/4
    (while that node is shallower than `cap`), else under a random node of
    depth < cap; paths reach the cap."""
    parent = np.full(n, -1, np.int32)
    depth = np.ones(n, np.int32)
    for i in range(1, n):
        if depth[i - 1] < cap and rng.random() < 0.75:
            parent[i] = i - 1
        else:
            open_nodes = np.flatnonzero(depth[:i] < cap)
            parent[i] = rng.choice(open_nodes) if open_nodes.size else -1
        depth[i] = 1 if parent[i] < 0 else depth[parent[i]] + 1
    return parent


def _deep_batch(seed, sizes, depth=32, hk=2, hv=4, fn=None):
    tb = _batch(seed, sizes, hk=hk, hv=hv, fn=fn or (lambda r, n: _deep_tree(r, n, depth)))
    tb.max_depth_bound = depth
    return tb


@pytest.mark.parametrize("sizes", [(128,), (128, 40, 1, 0, 77), (33, 32, 31, 128, 2)])
def test_deep_sizes(sizes):
    tb = _deep_batch(sum(sizes) + 7, sizes)
    depth = np.ones(tb.total_nodes, np.int64)
    for b in range(tb.batch):
        lo = tb.node_offsets[b]
        for i in range(tb.node_offsets[b + 1] - lo):
            a = tb.parent[lo + i]
            depth[lo + i] = 1 if a < 0 else depth[lo + a] + 1
    if max(sizes) >= 64:
        assert depth.max() > 16            # the paths go past the two-head kernel's bound
    o, status, _ = _verify(tb, max_depth=32)
    gb.check_status(status)
    assert _rel(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_deep_chains_and_general_kernel():
    # chains of 32 and 20 nodes and a random tree: paths up to the declared bound
    chains = {32: W.chain_tree(32), 20: W.chain_tree(20)}
    tb = _deep_batch(31, (32, 20, 128), fn=lambda r, n: chains[n] if n in chains else _deep_tree(r, n, 32))
    o, st, d = _verify(tb, max_depth=32)
    gb.check_status(st)
    o_gen, st2, _ = _verify(tb, d=d, max_depth=0)
    gb.check_status(st2)
    ref = oracle.verify(tb)
    assert _rel(o.float().cpu().numpy(), ref) <= TOL_BF16
    assert _rel(o_gen.float().cpu().numpy(), ref) <= TOL_BF16


def test_deep_tree_beyond_the_bound_is_flagged():
    tb = _deep_batch(32, (40, 30), fn=lambda r, n: W.chain_tree(n))
    out = torch.full((tb.total_nodes, tb.n_v_heads, tb.d_v), 7.0, dtype=torch.bfloat16, device="cuda")
    _, status, _ = _verify(tb, max_depth=32, out=out)
    assert int(status.item()) & DEV_TOO_DEEP
    assert torch.all(out[:40] == 7.0)          # the 40-deep chain is skipped
    assert _rel(out[40:].float().cpu().numpy(), oracle.verify(tb)[40:]) <= TOL_BF16


def test_deep_shallow_trees_under_a_deep_bound():
    # trees of depth <= 16 declared with max_depth 32 take the one-tile kernel
    tb = _batch(33, (128, 64, 100))
    tb.max_depth_bound = 32
    o, status, _ = _verify(tb, max_depth=32)
    gb.check_status(status)
    assert _rel(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_deep_fp32_output_many_items_and_S0_untouched():
    sizes = tuple((0, 1, 33, 128, 7, 100, 2, 128)[i % 8] for i in range(120))
    tb = _deep_batch(34, sizes)
    tb.scale = 0.5
    d = gb.upload(tb)
    before = d["S0"].clone()
    o, status, _ = _verify(tb, d=d, max_depth=32, out_dtype=torch.float32)
    gb.check_status(status)
    assert o.dtype == torch.float32
    assert torch.equal(before, d["S0"])
    assert _rel(o.cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_deep_non_finite_inputs_stay_on_their_branch():
    rng = np.random.default_rng(35)
    parent = _deep_tree(rng, 128, 32)
    base_tb = _deep_batch(35, (128,), hk=1, hv=2, fn=lambda r, n: parent)
    base, st, _ = _verify(base_tb, max_depth=32)
    gb.check_status(st)
    for bad_node in (0, 9, 100):
        sub = {bad_node}
        for i in range(128):
            if parent[i] in sub:
                sub.add(i)
        keep = [i for i in range(128) if i not in sub]
        tb2 = _deep_batch(35, (128,), hk=1, hv=2, fn=lambda r, n: parent)
        tb2.k[bad_node] = np.nan
        tb2.v[bad_node] = np.inf
        o2, st2, _ = _verify(tb2, max_depth=32)
        gb.check_status(st2)
        assert torch.equal(o2[keep], base[keep])


def test_deep_wait_probe_times_out_and_returns():
    tb = _deep_batch(36, (128, 50, 128))
    o0, st, d = _verify(tb, max_depth=32)
    gb.check_status(st)
    try:
        gb.gdn_test_set_wait_probe(2000)
        o1, st1, _ = _verify(tb, d=d, max_depth=32)
        bits = int(st1.item())
    finally:
        gb.gdn_test_set_wait_probe(0)
    assert bits == 16
    assert torch.equal(o1, o0)


# ----------------------------------------------------------------------------
# the tensor-core commit for accepted paths of 17 to 32 nodes (max_path <= 32)
# ----------------------------------------------------------------------------

TOL_STATE = 1e-4


def _commit(tb, d, max_path, out=None):
    status = gb.new_status()
    S = gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                           d["path_offsets"], d["path_idx"], tb.max_nodes, max_path=max_path, out=out,
                           dev_status=status)
    torch.cuda.synchronize()
    return S, status


@pytest.mark.parametrize("path", ["leaf", "deepest", "empty", "chain32"])
def test_long_path_commit_matches_oracle(path):
    fns = {"leaf": W.path_random_leaf, "deepest": W.path_deepest_leaf, "empty": lambda p, r: [],
           "chain32": W.path_whole_chain}
    rng = np.random.default_rng(41)
    if path == "chain32":
        parents = [W.chain_tree(32), W.chain_tree(17), W.chain_tree(1)]
    else:
        parents = [_deep_tree(rng, n, 32) for n in (128, 40, 1, 77)]
    tb = W.custom(41, parents, n_k_heads=2, n_v_heads=4, d=128, qkv_dtype="bf16", path_fn=fns[path])
    d = gb.upload(tb)
    S, status = _commit(tb, d, 32)
    gb.check_status(status)
    S_ref, st = oracle.commit(tb)
    assert st == 0
    assert _rel(S.cpu().numpy(), S_ref) <= TOL_STATE
    # the same as the general kernel (no declared bound)
    S_gen, status = _commit(tb, d, 0)
    gb.check_status(status)
    assert _rel(S_gen.cpu().numpy(), S_ref) <= TOL_STATE


def test_long_path_commit_in_place_and_many_items():
    rng = np.random.default_rng(42)
    parents = [_deep_tree(rng, int(n), 32) for n in rng.integers(20, 129, 150)]
    tb = W.custom(42, parents, n_k_heads=2, n_v_heads=4, d=128, qkv_dtype="bf16",
                  path_fn=W.path_deepest_leaf)
    d = gb.upload(tb)
    S_ref, st = oracle.commit(tb)
    assert st == 0
    S, status = _commit(tb, d, 32, out=d["S0"])
    gb.check_status(status)
    assert S.data_ptr() == d["S0"].data_ptr()
    assert _rel(S.cpu().numpy(), S_ref) <= TOL_STATE


def test_path_beyond_32_is_flagged():
    tb = W.custom(43, [W.chain_tree(40), W.chain_tree(30)], n_k_heads=1, n_v_heads=2, d=128,
                  qkv_dtype="bf16", path_fn=W.path_whole_chain)
    d = gb.upload(tb)
    sentinel = torch.full_like(d["S0"], 3.0)
    S, status = _commit(tb, d, 32, out=sentinel)
    assert int(status.item()) & DEV_TOO_DEEP
    assert torch.all(sentinel[0] == 3.0)       # the 40-node path is skipped
    S_ref, _ = oracle.commit(tb)
    assert _rel(sentinel[1].cpu().numpy(), S_ref[1]) <= TOL_STATE


def test_deep_commit_then_verify():
    # serving order on deep trees: the previous tree's accepted path (up to 32
    # nodes) committed on the tensor cores, the new tree verified from it
    prev, new = _deep_batch(44, (128, 90)), _deep_batch(45, (128, 100))
    dp, dn = gb.upload(prev), gb.upload(new)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(dn["parent"], dn["node_offsets"], new.max_nodes,
                                         dev_status=status)
    o, S = gb.gdn_tree_commit_verify(dp, dp["S0"], prev.max_nodes, 32, dn["q"], dn["k"], dn["v"],
                                     dn["g"], dn["beta"], dn["node_offsets"], dn["parent"], mask,
                                     depth, new.max_nodes, max_depth=32, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    S_ref, st = oracle.commit(prev)
    assert st == 0
    assert _rel(S.cpu().numpy(), S_ref) <= TOL_STATE
    new.S0 = S_ref.astype(np.float32)
    assert _rel(o.float().cpu().numpy(), oracle.verify(new)) <= TOL_BF16


# ----------------------------------------------------------------------------
# one tile, paths of 33 to 64 nodes (declared max_depth 33..64, N <= 128)
# ----------------------------------------------------------------------------

def test_chain64_bf16_d128():
    # the 64-node chain at d = 128 in bf16, with a deep tree and a single node
    chain = W.chain_tree(64)
    tb = _deep_batch(51, (64, 128, 1), depth=64,
                     fn=lambda r, n: chain if n == 64 else _deep_tree(r, n, 64))
    tb.max_depth_bound = 64
    o, status, d = _verify(tb, max_depth=64)
    gb.check_status(status)
    ref = oracle.verify(tb)
    assert _rel(o.float().cpu().numpy(), ref) <= TOL_BF16
    o_gen, st2, _ = _verify(tb, d=d, max_depth=0)
    gb.check_status(st2)
    assert _rel(o_gen.float().cpu().numpy(), ref) <= TOL_BF16


def test_depth64_many_items_fp32_output_and_flag():
    sizes = tuple((128, 0, 65, 7, 100, 1)[i % 6] for i in range(60))
    tb = _deep_batch(52, sizes, depth=64)
    tb.max_depth_bound = 64
    o, status, _ = _verify(tb, max_depth=64, out_dtype=torch.float32)
    gb.check_status(status)
    assert _rel(o.cpu().numpy(), oracle.verify(tb)) <= TOL_BF16
    # a 70-node chain under a declared bound of 64 is flagged and skipped
    tb2 = _deep_batch(53, (70, 40), depth=64, fn=lambda r, n: W.chain_tree(n))
    out = torch.full((tb2.total_nodes, tb2.n_v_heads, tb2.d_v), 7.0, dtype=torch.bfloat16, device="cuda")
    _, status2, _ = _verify(tb2, max_depth=64, out=out)
    assert int(status2.item()) & DEV_TOO_DEEP
    assert torch.all(out[:70] == 7.0)
    assert _rel(out[70:].float().cpu().numpy(), oracle.verify(tb2)[70:]) <= TOL_BF16


def test_depth64_non_finite_inputs_stay_on_their_branch():
    parent = W.chain_tree(64)
    parent[40] = 20                            # a branch at node 20: 40..63 hang under it
    base_tb = _deep_batch(54, (64,), hk=1, hv=2, depth=64, fn=lambda r, n: parent)
    base, st, _ = _verify(base_tb, max_depth=64)
    gb.check_status(st)
    for bad_node in (10, 45):
        sub = {bad_node}
        for i in range(64):
            if parent[i] in sub:
                sub.add(i)
        keep = [i for i in range(64) if i not in sub]
        tb2 = _deep_batch(54, (64,), hk=1, hv=2, depth=64, fn=lambda r, n: parent)
        tb2.k[bad_node] = np.nan
        tb2.g[bad_node] = np.inf
        o2, st2, _ = _verify(tb2, max_depth=64)
        gb.check_status(st2)
        assert torch.equal(o2[keep], base[keep])

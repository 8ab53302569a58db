"""GPU parity of gdn_tree_states: the state at chosen nodes.

The state at node i is the gated delta rule walked along i's root-to-node path
from S0 ("Trees from Marginals", gist.science Technical Summary, section 3,
Solution, bullet 4, applied to a node not yet accepted).  The oracle is
oracle.state_at (the plain float64 walk); tolerance 1e-4 * max|S| as for the
commit.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_net_gb300 import binding as gb
from gated_delta_net_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_STATE = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_net_gb300 import build
    build.build()
    gb.lib()


def _batch(seed, sizes, hk=2, hv=4):
    rng = np.random.default_rng(seed)
    parents = [np.zeros(0, np.int32) if n == 0 else W.chain_tree(n) if n == 16
               else W.depth_capped_random_tree(rng, n, 16) for n in sizes]
    return W.custom(seed, parents, n_k_heads=hk, n_v_heads=hv, d=128, qkv_dtype="bf16")


def _run(tb, d, sel_req, sel_node, out=None):
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    sr = torch.tensor(sel_req, dtype=torch.int32, device="cuda")
    sn = torch.tensor(sel_node, dtype=torch.int32, device="cuda")
    S = gb.gdn_tree_states(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                           mask, sr, sn, tb.max_nodes, out=out, dev_status=status)
    torch.cuda.synchronize()
    return S, status, mask


def _check_against_oracle(tb, S, sel_req, sel_node):
    got = S.cpu().numpy()
    for s, (b, i) in enumerate(zip(sel_req, sel_node)):
        for h in range(tb.n_v_heads):
            ref = oracle.state_at(tb, b, h, i)
            scale = max(float(np.max(np.abs(ref))), 1e-30)
            assert float(np.max(np.abs(got[s, h] - ref))) <= TOL_STATE * scale, (s, b, i, h)


def test_states_match_the_walked_state():
    tb = _batch(41, (128, 1, 16, 57, 0, 100))
    rng = np.random.default_rng(2)
    sel_req, sel_node = [], []
    for b in range(tb.batch):
        n = int(tb.node_offsets[b + 1] - tb.node_offsets[b])
        for i in ([0, n - 1] + list(rng.integers(0, n, 3)) if n else []):
            sel_req.append(b)
            sel_node.append(int(i))
    d = gb.upload(tb)
    S, status, _ = _run(tb, d, sel_req, sel_node)
    gb.check_status(status)
    _check_against_oracle(tb, S, sel_req, sel_node)


def test_state_at_the_accepted_leaf_equals_the_commit_bit_for_bit():
    tb = W.serving_target(batch=8)
    d = gb.upload(tb)
    sel_req = list(range(tb.batch))
    sel_node = [int(tb.path_idx[tb.path_offsets[b + 1] - 1]) for b in range(tb.batch)]
    S, status, _ = _run(tb, d, sel_req, sel_node)
    gb.check_status(status)
    st2 = gb.new_status()
    S_commit = gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                                  d["parent"], d["path_offsets"], d["path_idx"], tb.max_nodes,
                                  max_path=16, dev_status=st2)
    torch.cuda.synchronize()
    gb.check_status(st2)
    assert torch.equal(S, S_commit)


def test_many_selections_per_block_with_duplicates():
    tb = _batch(43, (128, 64, 128, 16))
    rng = np.random.default_rng(4)
    sizes = np.diff(tb.node_offsets)
    sel_req = [int(b) for b in rng.integers(0, tb.batch, 100)]
    sel_node = [int(rng.integers(0, sizes[b])) for b in sel_req]
    sel_req += sel_req[:5]
    sel_node += sel_node[:5]                     # the same node selected twice
    d = gb.upload(tb)
    S, status, _ = _run(tb, d, sel_req, sel_node)
    gb.check_status(status)
    assert torch.equal(S[:5], S[100:105])
    pick = list(range(0, 105, 7))
    _check_against_oracle(tb, S[pick], [sel_req[s] for s in pick], [sel_node[s] for s in pick])


def test_bad_selections_are_flagged_and_left_unwritten():
    tb = _batch(44, (40, 20))
    d = gb.upload(tb)
    out = torch.full((4, tb.n_v_heads, 128, 128), 3.0, device="cuda")
    S, status, _ = _run(tb, d, [0, 1, 5, 0], [3, 20, 0, 39], out=out)   # 20 is past request 1
    assert int(status.item()) == 2                                         # GDN_DEV_BAD_PATH
    assert torch.all(S[1] == 3.0) and torch.all(S[2] == 3.0)
    _check_against_oracle(tb, S[[0, 3]], [0, 0], [3, 39])


def test_stale_mask_row_and_deep_node():
    tb = W.custom(45, [W.chain_tree(20), W.depth_capped_random_tree(np.random.default_rng(1), 30, 16)],
                  n_k_heads=1, n_v_heads=2, d=128, qkv_dtype="bf16")
    d = gb.upload(tb)
    status = gb.new_status()
    mask, _ = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes, dev_status=status)
    lo = int(tb.node_offsets[1])
    mask[lo + 7, 0] ^= 1                        # node 7 of request 1: root bit flipped
    out = torch.full((2, 2, 128, 128), 3.0, device="cuda")
    gb.gdn_tree_states(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                       mask, torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                       torch.tensor([19, 7], dtype=torch.int32, device="cuda"), tb.max_nodes, out=out,
                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 8 | 32         # TOO_DEEP (20-node path) and BAD_DESC
    assert torch.all(out == 3.0)

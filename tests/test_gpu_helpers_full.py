"""The helper entry points at the sizes and launch configurations bench.py's
--helpers leg times (64 trees of 128 nodes, 16 key / 32 value heads, d = 128):

  * gdn_tree_relabel and gdn_gather_rows on the trees under random labels,
    bit-exact against oracle/relabel.py and plain indexing;
  * gdn_tree_grow with w = 1 and w = 8, bit-exact against oracle/grow.py;
  * gdn_tree_states at four candidate leaves per request: the accepted leaf's
    state equals the commit bit for bit, and sampled states match the walked
    state of the oracle (1e-4 of max|S|).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import grow as G
from oracle import relabel as R
from gated_delta_net_gb300 import binding as gb
from gated_delta_net_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_STATE = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_net_gb300 import build
    build.build()
    gb.lib()


@pytest.fixture(scope="module")
def tb():
    return W.serving_target()


def _shuffled_parents(tb, seed=5):
    rng = np.random.default_rng(seed)
    offs = tb.node_offsets.astype(np.int32)
    out = np.empty(tb.total_nodes, np.int32)
    for b in range(tb.batch):
        lo, hi = int(offs[b]), int(offs[b + 1])
        perm = rng.permutation(hi - lo)
        for i in range(hi - lo):
            p = int(tb.parent[lo + i])
            out[lo + perm[i]] = -1 if p < 0 else perm[p]
    return out


def test_relabel_and_gathers_full_size(tb):
    offs = tb.node_offsets.astype(np.int32)
    shuffled = _shuffled_parents(tb)
    status = gb.new_status()
    offs_d = torch.from_numpy(offs).cuda()
    order, rank, par_out = gb.gdn_tree_relabel(torch.from_numpy(shuffled).cuda(), offs_d, tb.max_nodes,
                                               dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    r_order, r_rank, r_par, bad = R.relabel(shuffled, offs)
    assert not np.any(bad)
    assert np.array_equal(order.cpu().numpy(), r_order)
    assert np.array_equal(rank.cpu().numpy(), r_rank)
    assert np.array_equal(par_out.cpu().numpy(), r_par)
    d = gb.upload(tb)
    glob = (np.repeat(offs[:-1], np.diff(offs)) + r_order).astype(np.int64)
    for key in ("q", "k", "v", "g", "beta"):
        out = gb.gdn_gather_rows(d[key], order, offs_d, dev_status=status)
        torch.cuda.synchronize()
        gb.check_status(status)
        assert torch.equal(out, d[key][torch.from_numpy(glob).cuda()]), key


@pytest.mark.parametrize("width", [1, 8])
def test_grow_full_size(tb, width):
    offs = tb.node_offsets.astype(np.int32)
    c, e = W.grow_draws(7, offs)
    status = gb.new_status()
    p, s, n = gb.gdn_tree_grow(torch.from_numpy(offs).cuda(), torch.from_numpy(c).cuda(),
                               torch.from_numpy(e).cuda(), width, 16, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    rp, rs, rn = G.grow(offs, width, 16, c, e)
    assert np.array_equal(n.cpu().numpy(), rn)
    assert np.array_equal(p.cpu().numpy(), rp)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_states_at_four_leaves_per_request_full_size(tb):
    offs = tb.node_offsets.astype(np.int32)
    leaves, first = [], []   # first: each request's accepted leaf, its first selection
    for b in range(tb.batch):
        lo, hi = int(offs[b]), int(offs[b + 1])
        par = tb.parent[lo:hi]
        has_child = np.zeros(hi - lo, bool)
        has_child[par[par >= 0]] = True
        cand = [int(tb.path_idx[tb.path_offsets[b + 1] - 1])]
        cand += [int(i) for i in np.flatnonzero(~has_child) if int(i) != cand[0]][:3]
        first.append(len(leaves))
        leaves += [(b, i) for i in cand]
    d = gb.upload(tb)
    status = gb.new_status()
    mask, _ = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes, dev_status=status)
    sr = torch.tensor([b for b, _ in leaves], dtype=torch.int32, device="cuda")
    sn = torch.tensor([i for _, i in leaves], dtype=torch.int32, device="cuda")
    S = gb.gdn_tree_states(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                           mask, sr, sn, tb.max_nodes, dev_status=status)
    S_commit = gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                                  d["path_offsets"], d["path_idx"], tb.max_nodes, max_path=16,
                                  dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    assert torch.equal(S[torch.tensor(first, device="cuda")], S_commit)
    got = S.cpu().numpy()
    rng = np.random.default_rng(3)
    for s in rng.choice(len(leaves), 12, replace=False):
        b, i = leaves[s]
        h = int(rng.integers(tb.n_v_heads))
        ref = oracle.state_at(tb, b, h, i)
        scale = max(float(np.max(np.abs(ref))), 1e-30)
        assert float(np.max(np.abs(got[s, h] - ref))) <= TOL_STATE * scale, (s, b, i, h)

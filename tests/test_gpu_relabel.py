"""GPU parity of the topological relabel and the row gather (integer work: bit-exact).

The relabel oracle is oracle/relabel.py (nodes by (depth, old id)); "Trees from
Marginals" (gist.science Technical Summary, section 3, Solution, bullet 1)
requires the topological order the relabel produces.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import relabel as R
from gated_delta_net_gb300 import binding as gb
from gated_delta_net_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_net_gb300 import build
    build.build()
    gb.lib()


def _shuffle_labels(parent, rng):
    """The same forest under a random labelling: returns (parent', perm) with
    perm[old] = new label."""
    n = len(parent)
    perm = rng.permutation(n)
    out = np.empty(n, np.int32)
    for i in range(n):
        out[perm[i]] = -1 if parent[i] < 0 else perm[parent[i]]
    return out, perm


def _batch(seed, sizes):
    rng = np.random.default_rng(seed)
    parents, offs = [], [0]
    for n in sizes:
        if n == 0:
            p = np.zeros(0, np.int32)
        elif n == 256:
            p = np.array([i + 1 for i in range(n - 1)] + [-1], np.int32)   # a chain, labelled backwards
        else:
            p, _ = _shuffle_labels(W.depth_capped_random_tree(rng, n, 16), rng)
        parents.append(p)
        offs.append(offs[-1] + n)
    return np.concatenate(parents).astype(np.int32), np.array(offs, np.int32)


@pytest.mark.parametrize("sizes", [(1,), (5, 0, 128, 33), (256, 7, 64), tuple(range(1, 60, 3))])
def test_relabel_bit_exact(sizes):
    parent, offs = _batch(sum(sizes), sizes)
    order, rank, parent_out, bad = R.relabel(parent, offs)
    assert not bad.any()
    status = gb.new_status()
    o, r, p = gb.gdn_tree_relabel(torch.from_numpy(parent).cuda(), torch.from_numpy(offs).cuda(),
                                  max(max(sizes), 1), dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    assert np.array_equal(o.cpu().numpy(), order)
    assert np.array_equal(r.cpu().numpy(), rank)
    assert np.array_equal(p.cpu().numpy(), parent_out)


@pytest.mark.parametrize("bad_parent", [[1, 0, -1], [-1, 1, 0], [-1, 7, 0], [-1, -3, 0]])
def test_malformed_request_is_flagged_and_left_untouched(bad_parent):
    good, offs_g = _batch(5, (40, 17))
    parent = np.concatenate([good[:40], np.array(bad_parent, np.int32), good[40:]])
    offs = np.array([0, 40, 40 + len(bad_parent), 40 + len(bad_parent) + 17], np.int32)
    status = gb.new_status()
    T = len(parent)
    outs = [torch.full((T,), -7, dtype=torch.int32, device="cuda") for _ in range(3)]
    par_d, offs_d = torch.from_numpy(parent).cuda(), torch.from_numpy(offs).cuda()   # held until the sync
    a = gb.lib().gdn_tree_relabel(gb._ptr(par_d), gb._ptr(offs_d), 3, T, 64, gb._ptr(outs[0]),
                                  gb._ptr(outs[1]), gb._ptr(outs[2]), gb._ptr(status), None)
    torch.cuda.synchronize()
    assert a == gb.GDN_OK
    assert int(status.item()) == 1
    ref = R.relabel(parent, offs)
    for got, want in zip(outs, ref[:3]):
        got = got.cpu().numpy()
        assert np.all(got[40:40 + len(bad_parent)] == -7)
        keep = np.r_[0:40, 40 + len(bad_parent):T]
        assert np.array_equal(got[keep], want[keep])


def test_gather_rows_bit_exact_and_bad_index():
    rng = np.random.default_rng(3)
    parent, offs = _batch(9, (50, 0, 128, 3))
    order, rank, _, _ = R.relabel(parent, offs)
    T = len(parent)
    src = torch.randn(T, 4, 24, device="cuda").to(torch.bfloat16)       # 192-byte rows
    idx = torch.from_numpy(order.astype(np.int32)).cuda()
    offs_d = torch.from_numpy(offs).cuda()
    status = gb.new_status()
    dst = gb.gdn_gather_rows(src, idx, offs_d, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    want = torch.empty_like(src)
    for b in range(len(offs) - 1):
        lo, hi = int(offs[b]), int(offs[b + 1])
        want[lo:hi] = src[lo + torch.from_numpy(order[lo:hi]).long().cuda()] if hi > lo else src[lo:hi]
    assert torch.equal(dst, want)
    back = gb.gdn_gather_rows(dst, torch.from_numpy(rank.astype(np.int32)).cuda(), offs_d)
    assert torch.equal(back, src)
    idx_bad = idx.clone()
    idx_bad[5] = 99                       # outside request 0's 50 nodes
    out = torch.zeros_like(src)
    gb.gdn_gather_rows(src, idx_bad, offs_d, out=out, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 32
    assert torch.all(out[5] == 0)


def test_relabel_gather_verify_end_to_end():
    # a topologically sorted batch, shown to the library under random labels:
    # relabel -> gather the token rows -> verify -> gather o back by rank equals
    # the oracle's outputs of the original labelling, node by node
    tb = W.serving_target(batch=4)
    rng = np.random.default_rng(11)
    T, offs = tb.total_nodes, tb.node_offsets.astype(np.int32)
    shuffled = np.empty(T, np.int32)
    where = np.empty(T, np.int64)           # original global row -> shuffled global row
    for b in range(tb.batch):
        lo, hi = int(offs[b]), int(offs[b + 1])
        p, perm = _shuffle_labels(tb.parent[lo:hi], rng)
        shuffled[lo:hi] = p
        where[lo:hi] = lo + perm
    d = gb.upload(tb)
    status = gb.new_status()
    offs_d = d["node_offsets"]
    inv = np.argsort(where)                 # shuffled row -> original row
    inv_d = torch.from_numpy(inv).cuda()
    rows = {k: d[k][inv_d].contiguous() for k in ("q", "k", "v", "g", "beta")}  # tokens in shuffled labels
    order, rank, parent_new = gb.gdn_tree_relabel(torch.from_numpy(shuffled).cuda(), offs_d, 128,
                                                  dev_status=status)
    sorted_rows = {k: gb.gdn_gather_rows(v, order, offs_d, dev_status=status) for k, v in rows.items()}
    mask, depth = gb.gdn_tree_build_desc(parent_new, offs_d, 128, dev_status=status)
    o_new = gb.gdn_tree_verify(sorted_rows["q"], sorted_rows["k"], sorted_rows["v"], sorted_rows["g"],
                               sorted_rows["beta"], d["S0"], offs_d, parent_new, mask, depth, 128,
                               max_depth=16, dev_status=status)
    o_shuf = gb.gdn_gather_rows(o_new, rank, offs_d, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    ref = oracle.verify(tb)                 # original labels
    got = o_shuf.float().cpu().numpy()[where]
    scale = float(np.max(np.abs(ref)))
    assert float(np.max(np.abs(got - ref))) <= 2e-2 * scale

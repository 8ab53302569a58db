"""GPU parity of gdn_tree_grow (top-w best-first construction): parent, score
and node counts bit-exact against oracle/grow.py (the modified DySpec search of
"Trees from Marginals", gist.science Technical Summary, Methodology, section 2)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import grow as G
from gated_delta_net_gb300 import binding as gb
from gated_delta_net_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_net_gb300 import build
    build.build()
    gb.lib()


def _run(caps, width, depth, seed, maxc=8, draws=None):
    offs = np.concatenate([[0], np.cumsum(caps)]).astype(np.int32)
    c, e = draws if draws is not None else W.grow_draws(seed, offs, maxc)
    status = gb.new_status()
    p, s, n = gb.gdn_tree_grow(torch.from_numpy(offs).cuda(), torch.from_numpy(c).cuda(),
                               torch.from_numpy(e).cuda(), width, depth, dev_status=status)
    torch.cuda.synchronize()
    return offs, c, e, p.cpu().numpy(), s.cpu().numpy(), n.cpu().numpy(), status


@pytest.mark.parametrize("caps,width,depth", [
    ((128,) * 4, 1, 16), ((128,) * 4, 8, 16), ((1, 2, 0, 17, 256), 2, 16), ((64, 100), 256, 16),
    ((90, 90, 90), 3, 3), ((50,), 1, 1)])
def test_grow_bit_exact(caps, width, depth):
    offs, c, e, p, s, n, status = _run(caps, width, depth, seed=sum(caps) + width)
    gb.check_status(status)
    rp, rs, rn = G.grow(offs, width, depth, c, e)
    assert np.array_equal(n, rn)
    assert np.array_equal(p, rp)
    assert np.array_equal(s.view(np.uint32), rs.view(np.uint32))   # bit-exact, -inf padding included


def test_grow_ties_and_clipped_children():
    caps = (60, 60)
    T = sum(caps)
    c = np.full(T, 2, np.int32)
    c[5] = 99                                  # clipped to max_children
    c[7] = -3                                  # clipped to 0
    e = np.ones((T, 4), np.float32)            # constant draws: many score ties
    offs, _, _, p, s, n, status = _run(caps, 3, 16, 0, draws=(c, e))
    gb.check_status(status)
    rp, rs, rn = G.grow(offs, 3, 16, c, e)
    assert np.array_equal(p, rp) and np.array_equal(n, rn)
    assert np.array_equal(s.view(np.uint32), rs.view(np.uint32))


def test_capacity_above_256_is_flagged():
    offs = np.array([0, 300], np.int32)
    c, e = W.grow_draws(1, offs)
    status = gb.new_status()
    gb.gdn_tree_grow(torch.from_numpy(offs).cuda(), torch.from_numpy(c).cuda(), torch.from_numpy(e).cuda(),
                     1, 16, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 4


def test_grown_trees_verify_against_the_oracle():
    # grow -> build_desc -> verify on the grown trees, against the float64 oracle
    caps = (128, 77, 128)
    offs, c, e, p, s, n, status = _run(caps, 4, 16, seed=9)
    gb.check_status(status)
    assert list(n) == list(caps)
    parents = [p[offs[b]:offs[b + 1]] for b in range(len(caps))]
    tb = W.custom(9, parents, n_k_heads=2, n_v_heads=4, d=128, qkv_dtype="bf16")
    d = gb.upload(tb)
    mask, depth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], 128, dev_status=status)
    o = gb.gdn_tree_verify(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                           d["parent"], mask, depth, 128, max_depth=16, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    ref = oracle.verify(tb)
    assert float(np.max(np.abs(o.float().cpu().numpy() - ref))) <= 2e-2 * float(np.max(np.abs(ref)))

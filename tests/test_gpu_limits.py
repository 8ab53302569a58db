"""GPU checks of the fast kernels' limits and failure reporting:

  * descriptor rows wider than the tensor-core verify reads (mask_words up to 8
    for trees of at most 128 nodes) verify like narrow ones, and a stray bit in
    the unread words is reported as a stale descriptor;
  * keys and queries far from unit norm (k_i . k_j beyond the fp16 range)
    match the oracle on the fast path as on the general one;
  * every bounded wait of the tensor-core verify and commit ends: the wait
    probe makes one wait run out, the kernels report GDN_DEV_TIMEOUT, return,
    and the results and the next launches are unchanged.

Reference: the float64 oracle ("Trees from Marginals", gist.science Technical
Summary, section 3 "Rollback-Free Tree Verification for GDN").
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_net_gb300 import binding as gb
from gated_delta_net_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_BF16, TOL_STATE = 2e-2, 1e-4
DEV_TIMEOUT, DEV_BAD_DESC = 16, 32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_net_gb300 import build
    build.build()
    gb.lib()
    yield
    gb.gdn_test_set_wait_probe(0)


def _rel(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-30)


def _tc_batch(seed, sizes, hk=2, hv=4):
    rng = np.random.default_rng(seed)
    parents = [W.depth_capped_random_tree(rng, n, 16) for n in sizes]
    tb = W.custom(seed, parents, n_k_heads=hk, n_v_heads=hv, d=128, qkv_dtype="bf16")
    tb.max_depth_bound = 16
    return tb


def _verify(tb, d, mask, depth, status, out=None, max_depth=16):
    o = gb.gdn_tree_verify(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                           d["parent"], mask, depth, tb.max_nodes, max_depth=max_depth,
                           scale=tb.scale, out=out, dev_status=status)
    torch.cuda.synchronize()
    return o


# ----------------------------------------------------------------------------
# descriptor rows of 5..8 words on the tensor-core path
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("words", [5, 8])
def test_wide_descriptor_rows_on_the_tc_path(words):
    tb = _tc_batch(71, (128, 97, 128, 33))
    d = gb.upload(tb)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes,
                                         mask_words=words, dev_status=status)
    narrow, ndepth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes,
                                            dev_status=status)
    o = _verify(tb, d, mask, depth, status)
    o_narrow = _verify(tb, d, narrow, ndepth, status)
    gb.check_status(status)
    assert mask.shape[1] == words
    assert torch.equal(o, o_narrow)
    assert _rel(o.float().cpu().numpy(), oracle.verify(tb)) <= TOL_BF16


def test_stray_bit_in_an_unread_word_is_a_stale_descriptor():
    tb = _tc_batch(72, (128, 64))
    d = gb.upload(tb)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes,
                                         mask_words=8, dev_status=status)
    torch.cuda.synchronize()
    gb.check_status(status)
    mask[5, 6] = 1                     # request 0, node 5: a bit for node 192
    out = torch.full((tb.total_nodes, tb.n_v_heads, tb.d_v), 3.0, dtype=torch.bfloat16,
                     device=d["q"].device)
    _verify(tb, d, mask, depth, status, out=out)
    assert int(status.item()) == DEV_BAD_DESC
    assert torch.all(out[:128] == 3.0)                 # the request is skipped
    ref = oracle.verify(tb)
    assert _rel(out[128:].float().cpu().numpy(), ref[128:]) <= TOL_BF16


# ----------------------------------------------------------------------------
# keys far from unit norm
# ----------------------------------------------------------------------------

def _large_key_batch(seed):
    """Keys of norm 300 that all point nearly the same way (k_i . k_j ~ 9e4,
    beyond fp16) with beta ~ 1e-6, so the recurrence stays tame
    (1 - beta |k|^2 ~ 0.9) and the exact outputs are moderate; queries of norm 40."""
    tb = _tc_batch(seed, (40, 64))
    rng = np.random.default_rng(seed)
    base = rng.standard_normal(128)
    base /= np.linalg.norm(base)
    for t in range(tb.total_nodes):
        for h in range(tb.n_k_heads):
            x = base + 0.05 * rng.standard_normal(128)
            tb.k[t, h] = W.round_to_bf16((300.0 * x / np.linalg.norm(x)).astype(np.float32))
            tb.q[t, h] = W.round_to_bf16(40.0 * tb.q[t, h])
    tb.beta[:] = 1.0e-6
    return tb


def test_unnormalised_keys_and_queries_match_the_oracle():
    tb = _large_key_batch(73)
    ref = oracle.verify(tb)
    assert np.all(np.isfinite(ref))
    d = gb.upload(tb)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes,
                                         dev_status=status)
    o = _verify(tb, d, mask, depth, status)
    gb.check_status(status)
    assert _rel(o.float().cpu().numpy(), ref) <= TOL_BF16
    # the general kernel (no declared depth bound) agrees
    o_gen = _verify(tb, d, mask, depth, status, max_depth=0)
    gb.check_status(status)
    assert _rel(o_gen.float().cpu().numpy(), ref) <= TOL_BF16


# ----------------------------------------------------------------------------
# bounded waits
# ----------------------------------------------------------------------------

def test_wait_probe_times_out_and_the_kernels_return():
    tb = _tc_batch(74, (128, 77, 128, 5, 128))
    d = gb.upload(tb)
    status = gb.new_status()
    mask, depth = gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes,
                                         dev_status=status)

    def run():
        o = _verify(tb, d, mask, depth, status)
        S = gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                               d["parent"], d["path_offsets"], d["path_idx"], tb.max_nodes,
                               max_path=16, dev_status=status)
        torch.cuda.synchronize()
        return o, S

    o0, S0 = run()
    gb.check_status(status)
    try:
        gb.gdn_test_set_wait_probe(2000)
        o1, S1 = run()
        bits = int(status.item())
    finally:
        gb.gdn_test_set_wait_probe(0)
    assert bits == DEV_TIMEOUT
    assert torch.equal(o1, o0) and torch.equal(S1, S0)
    # the context is still usable and the next launches are clean and identical
    status.zero_()
    o2, S2 = run()
    gb.check_status(status)
    assert torch.equal(o2, o0) and torch.equal(S2, S0)
    # the commit alone also reports the probe
    try:
        gb.gdn_test_set_wait_probe(2000)
        status.zero_()
        gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"],
                           d["parent"], d["path_offsets"], d["path_idx"], tb.max_nodes,
                           max_path=16, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == DEV_TIMEOUT
    finally:
        gb.gdn_test_set_wait_probe(0)
    S_ref, st = oracle.commit(tb)
    assert st == 0
    assert _rel(S0.cpu().numpy(), S_ref) <= TOL_STATE

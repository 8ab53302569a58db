"""The library on caller streams and inside CUDA graphs.

Every entry point is asynchronous on the caller's stream and allocates nothing,
so one decoding iteration (descriptor, verify, states, commit) can be captured
into a CUDA graph and replayed, and independent batches can run on concurrent
streams.  Both must give exactly the eager single-stream results.
"""
import numpy as np
import pytest
import torch

from gated_delta_net_gb300 import binding as gb
from gated_delta_net_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_net_gb300 import build
    build.build()
    gb.lib()


def _iteration(tb, d, mask, depth, o, S, S_sel, sel_req, sel_node, status, stream):
    gb.gdn_tree_build_desc(d["parent"], d["node_offsets"], tb.max_nodes, mask, depth, mask.shape[1],
                           status, stream)
    gb.gdn_tree_verify(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                       mask, depth, tb.max_nodes, max_depth=16, out=o, dev_status=status, stream=stream)
    gb.gdn_tree_states(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"], mask,
                       sel_req, sel_node, tb.max_nodes, out=S_sel, dev_status=status, stream=stream)
    gb.gdn_tree_commit(d["k"], d["v"], d["g"], d["beta"], d["S0"], d["node_offsets"], d["parent"],
                       d["path_offsets"], d["path_idx"], tb.max_nodes, max_path=16, out=S,
                       dev_status=status, stream=stream)


def _buffers(tb, dev):
    T = tb.total_nodes
    words = (tb.max_nodes + 31) // 32
    mask = torch.empty((T, words), dtype=torch.int32, device=dev)
    depth = torch.empty(T, dtype=torch.int32, device=dev)
    o = torch.empty((T, tb.n_v_heads, tb.d_v), dtype=torch.bfloat16, device=dev)
    S = torch.empty((tb.batch, tb.n_v_heads, tb.d_v, tb.d_k), dtype=torch.float32, device=dev)
    sel_req = torch.arange(tb.batch, dtype=torch.int32, device=dev)
    sel_node = torch.tensor([int(tb.path_idx[tb.path_offsets[b + 1] - 1]) for b in range(tb.batch)],
                            dtype=torch.int32, device=dev)
    S_sel = torch.empty_like(S)
    return mask, depth, o, S, S_sel, sel_req, sel_node


def test_one_iteration_captured_in_a_cuda_graph_replays_exactly():
    tb = W.serving_target(batch=6)
    dev = torch.device("cuda", 0)
    d = gb.upload(tb, device=dev)
    status = gb.new_status(dev)
    eager = _buffers(tb, dev)
    _iteration(tb, d, *eager, status, torch.cuda.current_stream())
    torch.cuda.synchronize()
    gb.check_status(status)
    bufs = _buffers(tb, dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _iteration(tb, d, *bufs, status, torch.cuda.current_stream())
    for _ in range(3):
        for t in (bufs[2], bufs[3], bufs[4]):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        gb.check_status(status)
        for got, want in zip(bufs[:5], eager[:5]):
            assert torch.equal(got, want)
    # the states at the accepted leaves are the commit, bit for bit
    assert torch.equal(bufs[4], bufs[3])


def test_independent_batches_on_concurrent_streams():
    dev = torch.device("cuda", 0)
    tbs = [W.serving_target(seed=s, batch=5) for s in (11, 12, 13)]
    runs = []
    for tb in tbs:
        d = gb.upload(tb, device=dev)
        runs.append((tb, d, _buffers(tb, dev), gb.new_status(dev)))
    # reference: one after another on the default stream
    refs = []
    for tb, d, bufs, st in runs:
        _iteration(tb, d, *bufs, st, torch.cuda.current_stream())
        torch.cuda.synchronize()
        refs.append([t.clone() for t in bufs[:5]])
        for t in bufs[2:5]:
            t.zero_()
    streams = [torch.cuda.Stream(dev) for _ in runs]
    torch.cuda.synchronize()
    for (tb, d, bufs, st), s in zip(runs, streams):
        _iteration(tb, d, *bufs, st, s)
    torch.cuda.synchronize()
    for (tb, d, bufs, st), ref in zip(runs, refs):
        gb.check_status(st)
        for got, want in zip(bufs[:5], ref):
            assert torch.equal(got, want)

"""Calls on several streams at once and calls replayed from a CUDA graph give the
bytes of the same calls issued one after another: the library keeps no state
between calls (a decode's work-item queue lives in its caller's workspace, the
prefill's work list in each CTA's shared memory).
"""
import math

import numpy as np
import pytest

from paged_kv_cache_wf_gb300 import binding as wf
from paged_kv_cache_wf_gb300 import workloads as W
from tests import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = G.torch_mod()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_cache_wf_gb300 import build
    build.build()


def _decode_inputs(lay, seed):
    torch = G.torch_mod()
    vals = W.draw_layer_values(lay, np.random.default_rng(seed))
    pools = G.build_dev_pools(lay, vals)
    g = lay.geom
    q = G.to_dev(vals.q, g.dtype)
    ws = torch.empty(max(16, wf.wf_paged_decode_workspace_size(lay.B, g.H_q, lay.max_seq_len,
                                                               wf.pool_desc(pools[0]))),
                     dtype=torch.uint8, device="cuda")
    bt = torch.from_numpy(lay.block_tables).cuda()
    sl = torch.from_numpy(lay.seq_lens).cuda()
    return dict(q=q, pools=pools, ws=ws, bt=bt, sl=sl, msl=lay.max_seq_len, scale=1.0 / math.sqrt(g.D))


def _decode(x, out, stream=None):
    kp, vp = x["pools"]
    wf.wf_paged_decode(out, x["q"], kp, vp, x["bt"], x["sl"], x["msl"], x["scale"], x["ws"], None,
                       stream.cuda_stream if stream is not None else None)


def test_decodes_on_four_streams_at_once_match_one_after_another():
    """Four decode batches (tensor-core kernel, several splits per sequence) issued
    concurrently on four streams, each with its own workspace."""
    torch = G.torch_mod()
    lays = [W.custom_layout(32, 8, 128, 16, W.BF16, [1, 300, 2049, 4100, 257], seed=60 + i) for i in range(2)]
    lays += [W.custom_layout(32, 8, 64, 16, W.BF16, [5, 700, 1500, 129], seed=62 + i) for i in range(2)]
    xs = [_decode_inputs(lay, 70 + i) for i, lay in enumerate(lays)]
    ref = []
    for x in xs:
        o = torch.empty_like(x["q"])
        _decode(x, o)
        ref.append(o)
    torch.cuda.synchronize()
    outs = [torch.full_like(x["q"], float("nan")) for x in xs]
    streams = [torch.cuda.Stream() for _ in xs]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for rep in range(3):
        for x, o, s in zip(xs, outs, streams):
            _decode(x, o, s)
    torch.cuda.synchronize()
    for o, r in zip(outs, ref):
        assert np.array_equal(G.storage_bytes(o), G.storage_bytes(r))


def test_prefill_and_decode_on_two_streams_match_one_after_another():
    """The persistent prefill grid on one stream beside a decode on another."""
    torch = G.torch_mod()
    pl = W.custom_layout(32, 8, 128, 16, W.BF16, [900, 1300, 257, 2049, 40], [300, 130, 257, 64, 40], seed=81)
    pv = W.draw_layer_values(pl, np.random.default_rng(82))
    ppools = G.build_dev_pools(pl, pv)
    x = _decode_inputs(W.custom_layout(32, 8, 128, 16, W.BF16, [3000, 17, 800], seed=83), 84)
    ref_p = G.run_prefill(pl, pv, ppools, 1.0 / math.sqrt(128))
    ref_d = torch.empty_like(x["q"])
    _decode(x, ref_d)
    torch.cuda.synchronize()
    kp, vp = ppools
    q = G.to_dev(pv.q, W.BF16)
    out_p = torch.full_like(q, float("nan"))
    out_d = torch.full_like(x["q"], float("nan"))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    bt, sl, cu = (torch.from_numpy(a).cuda() for a in (pl.block_tables, pl.seq_lens, pl.cu_q_lens))
    torch.cuda.synchronize()
    wf.wf_paged_prefill(out_p, q, kp, vp, bt, sl, cu, pl.max_q_len, pl.max_seq_len, 1.0 / math.sqrt(128), None,
                        s1.cuda_stream)
    _decode(x, out_d, s2)
    torch.cuda.synchronize()
    assert np.array_equal(G.storage_bytes(out_p), G.storage_bytes(ref_p))
    assert np.array_equal(G.storage_bytes(out_d), G.storage_bytes(ref_d))


def test_graph_replay_matches_eager_calls():
    """A scatter + decode + prefill sequence captured once as a CUDA graph: every
    replay writes the eager calls' bytes (the decode's queue is zeroed by a grid
    inside the graph, so replays do not depend on the previous one)."""
    torch = G.torch_mod()
    lay = W.custom_layout(32, 8, 128, 16, W.BF16, [1, 300, 2049, 4100, 257], seed=90)
    vals = W.draw_layer_values(lay, np.random.default_rng(91))
    x = _decode_inputs(lay, 91)
    kp, vp = x["pools"]
    g = lay.geom
    kn, vn = G.to_dev(vals.k_new, g.dtype), G.to_dev(vals.v_new, g.dtype)
    slots = torch.from_numpy(lay.new_slots()).cuda()
    pl = W.custom_layout(32, 8, 128, 16, W.BF16, [900, 1300, 257], [300, 130, 257], seed=92)
    pv = W.draw_layer_values(pl, np.random.default_rng(93))
    ppools = G.build_dev_pools(pl, pv)
    pq = G.to_dev(pv.q, W.BF16)
    pbt, psl, pcu = (torch.from_numpy(a).cuda() for a in (pl.block_tables, pl.seq_lens, pl.cu_q_lens))
    eager_d = torch.empty_like(x["q"])
    eager_p = torch.empty_like(pq)

    def step(out_d, out_p, stream):
        sp = stream.cuda_stream
        wf.wf_reshape_and_cache(kn, vn, kp, vp, slots, None, sp)
        _decode(x, out_d, stream)
        wf.wf_paged_prefill(out_p, pq, ppools[0], ppools[1], pbt, psl, pcu, pl.max_q_len, pl.max_seq_len,
                            1.0 / math.sqrt(128), None, sp)

    step(eager_d, eager_p, torch.cuda.current_stream())
    torch.cuda.synchronize()
    graph_d = torch.full_like(x["q"], float("nan"))
    graph_p = torch.full_like(pq, float("nan"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step(graph_d, graph_p, side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        graph_d.fill_(float("nan"))
        graph_p.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(G.storage_bytes(graph_d), G.storage_bytes(eager_d))
        assert np.array_equal(G.storage_bytes(graph_p), G.storage_bytes(eager_p))

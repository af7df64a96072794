"""The library's calls inside a CUDA graph: a serving engine captures its decode step
once and replays it.  The calls launch kernels only (no allocation, no
synchronisation, tensor maps encoded on the host), so a captured scatter + decode
(+ the copy-on-write copy) replays to the same bytes as the eager calls, for the
tensor-core paths (bf16 and fp8, whose grids are programmatic dependents of a
small preparing grid) and for the CUDA-core path."""
import math

import numpy as np
import pytest

import oracle
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


def _setup(H_q, H_kv, D, P, seqs, kv, seed):
    torch = G.torch_mod()
    lay = W.custom_layout(H_q, H_kv, D, P, W.BF16, seqs, seed=seed)
    vals = W.draw_layer_values(lay, np.random.default_rng(seed))
    g = lay.geom
    sc = dict(k_scale=1 / 64, v_scale=1 / 64) if kv == "fp8" else {}
    if kv == "fp8":
        kp = torch.full((g.N, g.P, g.H_kv, g.D), 0x7F, dtype=torch.uint8, device="cuda")
        vp = kp.clone()
    else:
        kp, vp = G.empty_dev_pool(g), G.empty_dev_pool(g)
    if vals.k_prefix.shape[0]:
        wf.wf_reshape_and_cache(G.to_dev(vals.k_prefix, W.BF16), G.to_dev(vals.v_prefix, W.BF16), kp, vp,
                                torch.from_numpy(lay.prefix_slots()).cuda(), None, None, **sc)
    dev = dict(q=G.to_dev(vals.q, W.BF16), k=G.to_dev(vals.k_new, W.BF16), v=G.to_dev(vals.v_new, W.BF16),
               slots=torch.from_numpy(lay.new_slots()).cuda(), bt=torch.from_numpy(lay.block_tables).cuda(),
               sl=torch.from_numpy(lay.seq_lens).cuda())
    ws = torch.empty(wf.wf_paged_decode_workspace_size(lay.B, g.H_q, lay.max_seq_len, wf.pool_desc(kp, **sc)),
                     dtype=torch.uint8, device="cuda")
    return lay, vals, kp, vp, dev, ws, sc


@pytest.mark.parametrize("H_q,H_kv,D,P,kv", [
    (32, 8, 128, 16, "bf16"),     # tensor-core decode (reset grid + split + combine)
    (32, 8, 128, 16, "fp8"),      # fp8 tensor-core decode (q prepare + split + combine)
    (8, 2, 64, 16, "bf16"),       # CUDA-core decode
])
def test_captured_step_replays_to_the_eager_bytes(H_q, H_kv, D, P, kv):
    torch = G.torch_mod()
    lay, vals, kp, vp, dev, ws, sc = _setup(H_q, H_kv, D, P, [700, 33, 129, 1, 2000], kv, seed=3)
    scale = 1.0 / math.sqrt(D)
    st = G.dev_status()
    kp0, vp0 = kp.clone(), vp.clone()

    def step(out, stream=None):
        wf.wf_reshape_and_cache(dev["k"], dev["v"], kp, vp, dev["slots"], st, stream, **sc)
        wf.wf_paged_decode(out, dev["q"], kp, vp, dev["bt"], dev["sl"], lay.max_seq_len, scale, ws, st, stream,
                           **sc)

    eager = torch.empty_like(dev["q"])
    step(eager)
    torch.cuda.synchronize()
    kp_eager, vp_eager = kp.clone(), vp.clone()
    # capture on a side stream, from the pools as they were before the step
    kp.copy_(kp0)
    vp.copy_(vp0)
    replay = torch.empty_like(dev["q"])
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step(replay)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for _ in range(3):                    # the scatter rewrites the same slots: replays are idempotent
        replay.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(G.storage_bytes(replay), G.storage_bytes(eager))
    assert np.array_equal(G.storage_bytes(kp), G.storage_bytes(kp_eager))
    assert np.array_equal(G.storage_bytes(vp), G.storage_bytes(vp_eager))
    assert wf.wf_device_status_fetch(st) == 0
    # and the replayed outputs are the right ones
    if kv == "bf16":
        kr, vr = oracle.build_pools(lay, vals)
        ref = oracle.paged_decode(vals.q, kr, vr, lay.block_tables, lay.seq_lens, scale, W.BF16)
        G.assert_close(G.from_dev(replay, W.BF16), ref, W.BF16, "graph replay")


def test_captured_copy_on_write_replays():
    torch = G.torch_mod()
    g = W.Geometry(H_q=8, H_kv=8, D=128, P=16, N=24, dtype=W.BF16)
    rng = np.random.default_rng(4)
    kh = W._draw(rng, (g.N, g.P, g.H_kv, g.D), g.dtype, 1.0)
    vh = W._draw(rng, (g.N, g.P, g.H_kv, g.D), g.dtype, 1.0)
    pairs = np.array([[3, 10], [5, 11], [7, 12]], np.int32)
    kp, vp = G.to_dev(kh, g.dtype), G.to_dev(vh, g.dtype)
    pr = torch.from_numpy(pairs).cuda()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            wf.wf_copy_blocks(kp, vp, pr)
    torch.cuda.current_stream().wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    oracle.copy_blocks(kh, vh, pairs, g.dtype)
    assert np.array_equal(G.storage_bytes(kp), kh.view(np.uint8).reshape(-1))
    assert np.array_equal(G.storage_bytes(vp), vh.view(np.uint8).reshape(-1))

"""The calls are stream-ordered and independent: a prefill and a decode that read the
same pool, issued on two streams after the step's scatter and running at the same
time, give byte for byte the outputs of the same calls run one after the other (the
way an engine overlaps the two halves of a mixed step), and both match the oracle.
"""
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


def test_prefill_and_decode_on_two_streams_match_the_sequential_run():
    torch = G.torch_mod()
    # requests with new rows (prefill) on cached prefixes; the decode reads the same
    # sequences with one query each
    seq_lens = [900, 1300, 257, 2049, 40, 700]
    q_lens = [300, 1, 257, 64, 40, 129]
    lay = W.custom_layout(32, 8, 128, 16, W.BF16, seq_lens, q_lens, seed=31)
    vals = W.draw_layer_values(lay, np.random.default_rng(32))
    g = lay.geom
    scale = 1.0 / math.sqrt(g.D)
    st = G.dev_status()
    kp, vp = G.build_dev_pools(lay, vals, st)
    q_pf = G.to_dev(vals.q, W.BF16)
    qd_host = W._draw(np.random.default_rng(33), (lay.B, g.H_q, g.D), W.BF16, 1.0)
    q_dec = G.to_dev(qd_host, W.BF16)
    bt = torch.from_numpy(lay.block_tables).cuda()
    sl = torch.from_numpy(lay.seq_lens).cuda()
    cu = torch.from_numpy(lay.cu_q_lens).cuda()
    ws = torch.empty(wf.wf_paged_decode_workspace_size(lay.B, g.H_q, lay.max_seq_len, wf.pool_desc(kp)),
                     dtype=torch.uint8, device="cuda")

    def prefill(out, stream=None):
        wf.wf_paged_prefill(out, q_pf, kp, vp, bt, sl, cu, lay.max_q_len, lay.max_seq_len, scale, st, stream)

    def decode(out, stream=None):
        wf.wf_paged_decode(out, q_dec, kp, vp, bt, sl, lay.max_seq_len, scale, ws, st, stream)

    seq_p, seq_d = torch.empty_like(q_pf), torch.empty_like(q_dec)
    prefill(seq_p)
    decode(seq_d)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        par_p, par_d = torch.full_like(q_pf, float("nan")), torch.full_like(q_dec, float("nan"))
        s1.wait_stream(torch.cuda.current_stream())
        s2.wait_stream(torch.cuda.current_stream())
        prefill(par_p, s1)
        decode(par_d, s2)
        torch.cuda.current_stream().wait_stream(s1)
        torch.cuda.current_stream().wait_stream(s2)
        torch.cuda.synchronize()
        assert np.array_equal(G.storage_bytes(par_p), G.storage_bytes(seq_p))
        assert np.array_equal(G.storage_bytes(par_d), G.storage_bytes(seq_d))
    assert wf.wf_device_status_fetch(st) == 0
    kh, vh = oracle.build_pools(lay, vals)
    ref_p = oracle.paged_prefill(vals.q, kh, vh, lay.block_tables, lay.seq_lens, lay.cu_q_lens, scale, W.BF16)
    ref_d = oracle.paged_decode(qd_host, kh, vh, lay.block_tables, lay.seq_lens, scale, W.BF16)
    G.assert_close(G.from_dev(seq_p, W.BF16), ref_p, W.BF16, "prefill")
    G.assert_close(G.from_dev(seq_d, W.BF16), ref_d, W.BF16, "decode")

"""wf_paged_prefill_decode: a mixed step's prefill and decode in one call (one grid
for the shapes both tensor-core kernels take).  Its outputs are byte for byte those
of wf_paged_prefill followed by wf_paged_decode on the same inputs, and both match
the fp64 oracle (tiny-vllm-py, "Inference Server Flow": a step mixes the two).
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


def _run_both_ways(pf_lay, dc_lay, kp, vp, q_pf, q_dec, scale, st):
    """(prefill, decode) outputs of the separate calls and of the one call."""
    torch = G.torch_mod()
    pbt, psl, pcu = (torch.from_numpy(x).cuda() for x in (pf_lay.block_tables, pf_lay.seq_lens, pf_lay.cu_q_lens))
    dbt, dsl = (torch.from_numpy(x).cuda() for x in (dc_lay.block_tables, dc_lay.seq_lens))
    g = pf_lay.geom
    ws = torch.full((max(16, wf.wf_paged_decode_workspace_size(dc_lay.B, g.H_q, dc_lay.max_seq_len,
                                                                 wf.pool_desc(kp))),), 0xFF,
                    dtype=torch.uint8, device="cuda")     # dirty on purpose: needs no initialisation
    sep_p, sep_d = torch.full_like(q_pf, float("nan")), torch.full_like(q_dec, float("nan"))
    wf.wf_paged_prefill(sep_p, q_pf, kp, vp, pbt, psl, pcu, pf_lay.max_q_len, pf_lay.max_seq_len, scale, st)
    wf.wf_paged_decode(sep_d, q_dec, kp, vp, dbt, dsl, dc_lay.max_seq_len, scale, ws, st)
    one_p, one_d = torch.full_like(q_pf, float("nan")), torch.full_like(q_dec, float("nan"))
    wf.wf_paged_prefill_decode(one_p, q_pf, pbt, psl, pcu, pf_lay.max_q_len, pf_lay.max_seq_len, one_d, q_dec,
                               dbt, dsl, dc_lay.max_seq_len, kp, vp, scale, ws, st)
    return (sep_p, sep_d), (one_p, one_d)


@pytest.mark.parametrize("H_q,H_kv,D,P", [(32, 8, 128, 16), (16, 8, 64, 16), (8, 8, 128, 32),
                                          (16, 2, 128, 16)])   # the last: a group of 8, two launches
def test_one_call_equals_the_two_calls_and_the_oracle(H_q, H_kv, D, P):
    """Prefill requests with cached prefixes, and decodes of the same sequences (one
    query each) over the one pool."""
    seq_lens = [900, 1300, 257, 2049, 40, 700, 5]
    q_lens = [300, 1, 257, 64, 40, 129, 5]
    lay = W.custom_layout(H_q, H_kv, D, P, W.BF16, seq_lens, q_lens, seed=71)
    vals = W.draw_layer_values(lay, np.random.default_rng(72))
    g = lay.geom
    scale = 1.0 / math.sqrt(g.D)
    st = G.dev_status()
    kp, vp = G.build_dev_pools(lay, vals, st)
    q_pf = G.to_dev(vals.q, W.BF16)
    qd_host = W._draw(np.random.default_rng(73), (lay.B, g.H_q, g.D), W.BF16, 1.0)
    q_dec = G.to_dev(qd_host, W.BF16)
    (sep_p, sep_d), (one_p, one_d) = _run_both_ways(lay, lay, kp, vp, q_pf, q_dec, scale, st)
    assert wf.wf_device_status_fetch(st) == 0
    assert np.array_equal(G.storage_bytes(one_p), G.storage_bytes(sep_p))
    assert np.array_equal(G.storage_bytes(one_d), G.storage_bytes(sep_d))
    kh, vh = oracle.build_pools(lay, vals)
    ref_p = oracle.paged_prefill(vals.q, kh, vh, lay.block_tables, lay.seq_lens, lay.cu_q_lens, scale, W.BF16)
    ref_d = oracle.paged_decode(qd_host, kh, vh, lay.block_tables, lay.seq_lens, scale, W.BF16)
    G.assert_close(G.from_dev(one_p, W.BF16), ref_p, W.BF16, "prefill part")
    G.assert_close(G.from_dev(one_d, W.BF16), ref_d, W.BF16, "decode part")


def test_mixed_step_full_size_bytes_equal_the_two_calls():
    """The mixed continuous-batching step at Llama-3-8B shapes (8 prefills of
    128..2048 new tokens on prefixes of 0..2048, 120 decodes of 256..8192 positions,
    one churned pool), one layer: the one call gives the bytes of the two calls."""
    torch = G.torch_mod()
    pf, dc = W.mixed_step(0)
    g = pf.geom
    kp, vp = W.device_pools([pf, dc], seed=81)
    pq, pk, pv = W.device_step_values(pf, seed=82)
    dq, dk, dv = W.device_step_values(dc, seed=83)
    st = G.dev_status()
    slots = torch.from_numpy(np.concatenate([pf.new_slots(), dc.new_slots()])).cuda()
    wf.wf_reshape_and_cache(torch.cat([pk, dk]), torch.cat([pv, dv]), kp, vp, slots, st)
    assert wf.wf_paged_prefill_decode_fused(wf.pool_desc(kp), g.H_q)
    (sep_p, sep_d), (one_p, one_d) = _run_both_ways(pf, dc, kp, vp, pq, dq, 1.0 / math.sqrt(g.D), st)
    assert wf.wf_device_status_fetch(st) == 0
    assert np.array_equal(G.storage_bytes(one_p), G.storage_bytes(sep_p))
    assert np.array_equal(G.storage_bytes(one_d), G.storage_bytes(sep_d))
    assert torch.isfinite(one_p.float()).all() and torch.isfinite(one_d.float()).all()


def test_empty_halves():
    """No prefill rows: the call is the decode; no decode sequence: the prefill."""
    torch = G.torch_mod()
    lay = W.custom_layout(32, 8, 128, 16, W.BF16, [300, 77], [100, 77], seed=91)
    vals = W.draw_layer_values(lay, np.random.default_rng(92))
    st = G.dev_status()
    kp, vp = G.build_dev_pools(lay, vals, st)
    q_pf = G.to_dev(vals.q, W.BF16)
    q_dec = G.to_dev(W._draw(np.random.default_rng(93), (lay.B, 32, 128), W.BF16, 1.0), W.BF16)
    bt, sl, cu = (torch.from_numpy(x).cuda() for x in (lay.block_tables, lay.seq_lens, lay.cu_q_lens))
    ws = torch.empty(wf.wf_paged_decode_workspace_size(lay.B, 32, lay.max_seq_len, wf.pool_desc(kp)),
                     dtype=torch.uint8, device="cuda")
    ref_d = torch.empty_like(q_dec)
    wf.wf_paged_decode(ref_d, q_dec, kp, vp, bt, sl, lay.max_seq_len, 0.088, ws, st)
    ref_p = torch.empty_like(q_pf)
    wf.wf_paged_prefill(ref_p, q_pf, kp, vp, bt, sl, cu, lay.max_q_len, lay.max_seq_len, 0.088, st)
    # decode only: a prefill batch with no rows
    no_q = q_pf[:0]
    zero_cu = torch.zeros(lay.B + 1, dtype=torch.int32, device="cuda")
    out_d = torch.empty_like(q_dec)
    wf.wf_paged_prefill_decode(no_q, no_q, bt, sl, zero_cu, 0, lay.max_seq_len, out_d, q_dec, bt, sl,
                               lay.max_seq_len, kp, vp, 0.088, ws, st)
    assert np.array_equal(G.storage_bytes(out_d), G.storage_bytes(ref_d))
    # prefill only: a decode batch of no sequences
    out_p = torch.empty_like(q_pf)
    wf.wf_paged_prefill_decode(out_p, q_pf, bt, sl, cu, lay.max_q_len, lay.max_seq_len, q_dec[:0], q_dec[:0],
                               bt[:0], sl[:0], lay.max_seq_len, kp, vp, 0.088, ws, st)
    assert np.array_equal(G.storage_bytes(out_p), G.storage_bytes(ref_p))
    assert wf.wf_device_status_fetch(st) == 0

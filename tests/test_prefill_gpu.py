"""wf_paged_prefill (tcgen05 tensor-core path) on the GPU against the fp64 oracle.

bf16 KV, fp32 accumulation: max abs <= 2e-2 and mean abs <= 2e-3.
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


CASES = {
    # H_q, H_kv, D, P, seq_lens, q_lens
    "no_prefix_one_tile": (8, 2, 128, 16, [100], [100]),
    "prefix_and_ragged": (8, 2, 128, 16, [20, 33, 300, 5], [20, 12, 170, 1]),
    "multi_q_tiles": (4, 4, 128, 16, [700, 260], [520, 129]),
    "long_prefix": (8, 1, 128, 7, [1500, 140], [33, 128]),
    "D64_gqa4": (16, 4, 64, 16, [400, 90, 1], [256, 90, 1]),
    "P1_P3_odd": (6, 3, 128, 3, [129, 257], [129, 2]),
    "gqa8": (16, 2, 128, 64, [333, 64], [200, 64]),
    "empty_request_in_batch": (4, 2, 128, 16, [50, 60, 70], [10, 0, 70]),
    # D = 64 instances of the pipelined tensor-core kernel at every group size
    "D64_mha_gpt2": (12, 12, 64, 16, [300, 129, 40], [300, 64, 40]),
    "D64_gqa2": (16, 8, 64, 16, [520, 77], [260, 77]),
    "D64_gqa8": (16, 2, 64, 32, [333, 64, 1], [200, 64, 1]),
    # large blocks, up to the largest block size the calls accept (1024 positions)
    "P256_gqa4": (32, 8, 128, 256, [700, 300, 1], [300, 128, 1]),
    "P1024_D64_gqa2": (16, 8, 64, 1024, [1500, 90], [700, 90]),
}


def _lengths(seed, B, q_lo, q_hi, c_lo, c_hi):
    rng = np.random.default_rng(seed)
    q = rng.integers(q_lo, q_hi + 1, size=B)
    c = rng.integers(c_lo, c_hi + 1, size=B)
    return list(map(int, q + c)), list(map(int, q))


# Work-list cases of the persistent grid (each CTA runs a longest-first list of query
# blocks): requests shorter than one query tile (items whose second tile is empty),
# many items per CTA with prefixes of every length, and a batch past the list build's
# request limit, which takes the one-CTA-per-block grid.
_SQ, _QL = _lengths(5, 40, 1, 31, 0, 600)
CASES["short_requests_many"] = (8, 2, 128, 16, _SQ, _QL)
_SQ, _QL = _lengths(6, 24, 100, 260, 0, 900)
CASES["several_blocks_per_cta"] = (32, 8, 128, 16, _SQ, _QL)
_SQ, _QL = _lengths(7, 1030, 1, 1, 0, 40)
CASES["requests_past_list_limit"] = (8, 2, 64, 16, _SQ, _QL)


# Every (D, G) instance of the one-CTA-per-query-block grid, which the standalone call
# takes past the persistent grid's list limits (here: more than 1024 requests).
LEGACY_GRID = [(64, 1), (64, 2), (64, 4), (64, 8), (128, 1), (128, 2), (128, 4), (128, 8)]


def _oracle_prefill(lay, vals, scale):
    kp, vp = oracle.build_pools(lay, vals)
    return oracle.paged_prefill(vals.q, kp, vp, lay.block_tables, lay.seq_lens, lay.cu_q_lens, scale,
                                lay.geom.dtype)


@pytest.mark.parametrize("name", list(CASES.keys()))
def test_prefill_matches_oracle(name):
    H_q, H_kv, D, P, sl, ql = CASES[name]
    lay = W.custom_layout(H_q, H_kv, D, P, W.BF16, sl, ql, seed=len(name))
    vals = W.draw_layer_values(lay, np.random.default_rng(41))
    scale = 1.0 / math.sqrt(D)
    st = G.dev_status()
    pools = G.build_dev_pools(lay, vals, st)
    out = G.run_prefill(lay, vals, pools, scale, st)
    got = G.from_dev(out, W.BF16)
    ref = _oracle_prefill(lay, vals, scale)
    G.assert_close(got, ref, W.BF16, name)
    assert wf.wf_device_status_fetch(st) == 0


def test_prefill_last_row_matches_decode_kernel():
    """The last prefill row of a request and a decode over the same cache agree."""
    lay = W.custom_layout(8, 2, 128, 16, W.BF16, [300, 77], [40, 77], seed=3)
    vals = W.draw_layer_values(lay, np.random.default_rng(3))
    pools = G.build_dev_pools(lay, vals)
    pre = G.from_dev(G.run_prefill(lay, vals, pools, 0.088), W.BF16)
    last = lay.cu_q_lens[1:] - 1
    dl = W.Layout(lay.geom, lay.seq_lens, np.ones(2, np.int32), lay.block_tables, lay.spare_block)
    dv = W.LayerValues(q=vals.q[last], k_new=vals.k_new[last], v_new=vals.v_new[last],
                       k_prefix=vals.k_prefix, v_prefix=vals.v_prefix)
    dec = G.from_dev(G.run_decode(dl, dv, pools, 0.088), W.BF16)
    assert np.abs(pre[last] - dec).max() <= 2e-2


def test_prefill_mixed_step_full_size_sampled():
    """Config 'mixed' prefill part at full size on the device; sampled query rows are
    recomputed by the oracle as decode rows at the row's causal length."""
    torch = G.torch_mod()
    pf, dc = W.mixed_step(0)
    g = pf.geom
    kp, vp = W.device_pools([pf, dc], seed=51)
    q, k_new, v_new = W.device_step_values(pf, seed=52)
    rng = np.random.default_rng(5)
    rows = []  # (request, row)
    for b in range(pf.B):
        n = int(pf.q_lens[b])
        picks = {0, n - 1, min(127, n - 1), min(128, n - 1)} | set(rng.integers(0, n, 3).tolist())
        rows += [(b, int(i)) for i in sorted(picks)]
    seqs = sorted({b for b, _ in rows})
    # host copies of the blocks these requests use, before the GPU scatter
    nb = [-(-int(pf.seq_lens[b]) // g.P) for b in seqs]
    used = np.unique(np.concatenate([pf.block_tables[b, :n] for b, n in zip(seqs, nb)]))
    remap = {int(x): i for i, x in enumerate(used)}
    idx = torch.from_numpy(used.astype(np.int64)).cuda()
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    hk, hv = bits(kp.index_select(0, idx)), bits(vp.index_select(0, idx))
    st = G.dev_status()
    wf.wf_reshape_and_cache(k_new, v_new, kp, vp, torch.from_numpy(pf.new_slots()).cuda(), st)
    out = torch.empty_like(q)
    wf.wf_paged_prefill(out, q, kp, vp, torch.from_numpy(pf.block_tables).cuda(),
                        torch.from_numpy(pf.seq_lens).cuda(), torch.from_numpy(pf.cu_q_lens).cuda(),
                        pf.max_q_len, pf.max_seq_len, 1 / math.sqrt(g.D), st)
    assert wf.wf_device_status_fetch(st) == 0
    assert torch.isfinite(out.float()).all()
    # oracle side: its own scatter of the new rows into the host sub-pool
    M = max(nb)
    hbt = np.zeros((len(seqs), M), np.int32)
    for i, (b, n) in enumerate(zip(seqs, nb)):
        hbt[i, :n] = [remap[int(x)] for x in pf.block_tables[b, :n]]
    cu = pf.cu_q_lens
    new_rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in seqs])
    sub = W.Layout(W.Geometry(g.H_q, g.H_kv, g.D, g.P, hk.shape[0], g.dtype), pf.seq_lens[seqs],
                   pf.q_lens[seqs], hbt, 0)
    oracle.reshape_and_cache(bits(k_new[new_rows]), bits(v_new[new_rows]), hk, hv, sub.new_slots(), g.dtype)
    # each sampled row = a decode row over positions 0 .. c_b + i
    pos = {b: i for i, b in enumerate(seqs)}
    qrows = np.array([cu[b] + i for b, i in rows])
    lens = np.array([int(pf.prefix_lens[b]) + i + 1 for b, i in rows], np.int32)
    tabs = np.stack([hbt[pos[b]] for b, _ in rows])
    ref = oracle.paged_decode(bits(q[qrows]), hk, hv, tabs, lens, 1 / math.sqrt(g.D), g.dtype)
    got = G.from_dev(out[qrows], g.dtype)
    G.assert_close(got, ref, g.dtype, "mixed prefill sample")


def test_prefill_flags_bad_lengths():
    torch = G.torch_mod()
    lay = W.custom_layout(4, 2, 128, 16, W.BF16, [40, 50], [10, 50], seed=6)
    vals = W.draw_layer_values(lay, np.random.default_rng(6))
    pools = G.build_dev_pools(lay, vals)
    bad = W.Layout(lay.geom, np.array([40, 20], np.int32), lay.q_lens, lay.block_tables, lay.spare_block)
    st = G.dev_status()
    q = G.to_dev(vals.q, W.BF16)
    out = torch.zeros_like(q)
    wf.wf_paged_prefill(out, q, pools[0], pools[1], torch.from_numpy(bad.block_tables).cuda(),
                        torch.from_numpy(bad.seq_lens).cuda(), torch.from_numpy(lay.cu_q_lens).cuda(),
                        50, 50, 0.1, st)
    assert wf.wf_device_status_fetch(st) == wf.WF_DEV_BAD_SEQLEN   # request 1: seq_len 20 < q_len 50
    ref = _oracle_prefill(lay, vals, 0.1)
    got = G.from_dev(out, W.BF16)
    G.assert_close(got[:10], ref[:10], W.BF16, "request 0 unaffected")


def legacy_grid_layout(D, grp):
    """1030 requests (past the persistent grid's request limit) of 1-3 new tokens on
    cached prefixes of 0..40 positions."""
    H_kv = 2
    sl, ql = _lengths(100 + D + grp, 1030, 1, 3, 0, 40)
    return W.custom_layout(grp * H_kv, H_kv, D, 16, W.BF16, sl, ql, seed=D * grp)


@pytest.mark.parametrize("D,grp", LEGACY_GRID)
def test_prefill_one_cta_per_block_grid(D, grp):
    """Every (D, G) instance of the per-block grid on a batch past the list limits."""
    lay = legacy_grid_layout(D, grp)
    assert not G.prefill_persistent(lay)
    vals = W.draw_layer_values(lay, np.random.default_rng(D + grp))
    scale = 1.0 / math.sqrt(D)
    st = G.dev_status()
    pools = G.build_dev_pools(lay, vals, st)
    got = G.from_dev(G.run_prefill(lay, vals, pools, scale, st), W.BF16)
    G.assert_close(got, _oracle_prefill(lay, vals, scale), W.BF16, f"per-block grid D={D} G={grp}")
    assert wf.wf_device_status_fetch(st) == 0

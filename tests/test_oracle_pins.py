"""Pins for the fp64 oracle: checks against things other than itself.

- worked paging examples printed on the pages (tests/golden/paging_examples.json);
- hand-derived closed forms (tests/golden/closed_form.json);
- a contiguous-cache brute force (tests/_brute.py) and torch SDPA in float64;
- the invariants ember's test suite pins: block-size invariance for
  P in {1, 2, 3, 7, 16, 64} and batch invariance ("Correctness");
- special cases: all keys equal -> mean of V, one position -> V[0],
  q = 0 -> mean of V, GQA == MHA with repeated KV heads, the last prefill row ==
  decode at the same length, pool relabelling.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_wf_gb300 import workloads as W
from tests._brute import brute_attention

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run_decode(layout, vals, scale, pools=None, nthreads=4):
    kp, vp = pools if pools is not None else oracle.build_pools(layout, vals)
    return oracle.paged_decode(vals.q, kp, vp, layout.block_tables, layout.seq_lens, scale,
                               layout.geom.dtype, nthreads)


def run_prefill(layout, vals, scale, pools=None, nthreads=4):
    kp, vp = pools if pools is not None else oracle.build_pools(layout, vals)
    return oracle.paged_prefill(vals.q, kp, vp, layout.block_tables, layout.seq_lens,
                                layout.cu_q_lens, scale, layout.geom.dtype, nthreads)


# --------------------------------------------------------------------------
# worked examples from the pages
# --------------------------------------------------------------------------
def _paging_examples():
    with open(os.path.join(GOLDEN, "paging_examples.json")) as f:
        return json.load(f)["examples"]


@pytest.mark.parametrize("ex", _paging_examples(), ids=lambda e: e["cite"][:20])
def test_paging_example_scatter_lands_where_the_page_says(ex):
    """Rows written through slot_mapping land in the (block, offset) the figure prints."""
    P = ex["block_size"]
    N = max(ex["block_table"]) + 2
    H_kv, D = 1, 4
    L = ex["length"]
    geom = W.Geometry(H_q=1, H_kv=H_kv, D=D, P=P, N=N, dtype=W.F32)
    bt = np.array([ex["block_table"]], dtype=np.int32)
    lay = W.Layout(geom, np.array([L], np.int32), np.array([L], np.int32), bt, N - 1)
    slots = lay.new_slots()                      # runner bookkeeping from the generator
    rows = np.zeros((L, H_kv, D), np.float32)
    rows[:, 0, 0] = np.arange(1, L + 1)          # row p carries the value p+1
    kp = W.empty_pool(geom)
    vp = W.empty_pool(geom)
    oracle.reshape_and_cache(rows, rows, kp, vp, slots, W.F32)
    for pos, blk, off in ex["expected"]:
        assert kp[blk, off, 0, 0] == pos + 1
        assert vp[blk, off, 0, 0] == pos + 1
    written = sum(1 for _ in ex["expected"])
    assert np.count_nonzero(~np.isnan(kp[:, :, 0, 0])) == written


@pytest.mark.parametrize("ex", _paging_examples(), ids=lambda e: e["cite"][:20])
def test_paging_example_gather_reads_where_the_page_says(ex):
    """Decode gathers position j from the figure's (block, offset): one-hot keys make
    the softmax pick position j, so the output is the V stored there."""
    P = ex["block_size"]
    N = max(ex["block_table"]) + 2
    L = ex["length"]
    D = max(L, 4)
    geom = W.Geometry(H_q=1, H_kv=1, D=D, P=P, N=N, dtype=W.F32)
    kp = W.empty_pool(geom)
    vp = W.empty_pool(geom)
    for pos, blk, off in ex["expected"]:       # place rows by the printed mapping only
        kp[blk, off, 0, :] = 0.0
        kp[blk, off, 0, pos] = 1.0
        vp[blk, off, 0, :] = 0.0
        vp[blk, off, 0, 0] = 100.0 + pos
    bt = np.array([ex["block_table"]], dtype=np.int32)
    for j in range(L):
        q = np.zeros((1, 1, D), np.float32)
        q[0, 0, j] = 1.0
        out = oracle.paged_decode(q, kp, vp, bt, np.array([L], np.int32), 200.0, W.F32, 1)
        assert abs(out[0, 0, 0] - (100.0 + j)) < 1e-9


def test_closed_form_golden():
    with open(os.path.join(GOLDEN, "closed_form.json")) as f:
        cases = json.load(f)["cases"]
    D = 64
    for c in cases:
        L = len(c["k"])
        geom = W.Geometry(H_q=1, H_kv=1, D=D, P=2, N=L + 2, dtype=W.F32)
        kp = W.empty_pool(geom)
        vp = W.empty_pool(geom)
        k = np.zeros((L, 1, D), np.float64)
        v = np.zeros((L, 1, D), np.float64)
        k[:, 0, :2] = c["k"]
        v[:, 0, :2] = c["v"]
        bt = np.array([list(range(L // 2 + 1))], np.int32)
        lay = W.Layout(geom, np.array([L], np.int32), np.array([L], np.int32), bt, L + 1)
        oracle.reshape_and_cache(k.astype(np.float32), v.astype(np.float32), kp, vp,
                                 lay.new_slots(), W.F32)
        q = np.zeros((1, 1, D), np.float64)
        q[0, 0, :2] = c["q"]
        out = oracle.paged_decode(q.astype(np.float32), kp, vp, bt, np.array([L], np.int32),
                                  c["scale"], W.F32, 1)
        # q rounded to float32 (relative 6e-8) is the only inexact input
        np.testing.assert_allclose(out[0, 0, :2], c["out"], rtol=0, atol=1e-6)
        assert np.all(out[0, 0, 2:] == 0.0)


# --------------------------------------------------------------------------
# brute force and library cross-checks
# --------------------------------------------------------------------------
SMALL = [
    # H_q, H_kv, D, P, dtype, seq_lens, q_lens
    (4, 2, 64, 16, W.F32, [6, 18, 34, 65], None),
    (8, 2, 64, 3, W.BF16, [1, 7, 20, 40], None),
    (4, 4, 128, 7, W.F32, [9, 15, 2], None),
    (8, 1, 64, 1, W.BF16, [5, 3], None),
    (4, 2, 64, 16, W.BF16, [20, 33, 5], [20, 12, 5]),     # prefill, with and without prefix
    (6, 3, 128, 5, W.F32, [11, 8], [4, 8]),
]


@pytest.mark.parametrize("case", SMALL)
def test_oracle_matches_contiguous_brute_force(case):
    H_q, H_kv, D, P, dt, sl, ql = case
    lay = W.custom_layout(H_q, H_kv, D, P, dt, sl, ql, seed=3)
    vals = W.draw_layer_values(lay, np.random.default_rng(11))
    scale = 1.0 / math.sqrt(D)
    ref = brute_attention(lay, vals, scale)
    if ql is None:
        got = run_decode(lay, vals, scale)
    else:
        got = run_prefill(lay, vals, scale)
    np.testing.assert_allclose(got.reshape(ref.shape), ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_oracle_matches_torch_sdpa_float64(causal):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    H_q, H_kv, D, P = 8, 2, 64, 5
    sl = [13, 30, 7]
    ql = [5, 30, 1] if causal else None
    lay = W.custom_layout(H_q, H_kv, D, P, W.BF16, sl, ql, seed=5)
    vals = W.draw_layer_values(lay, np.random.default_rng(2))
    scale = 0.11
    got = run_prefill(lay, vals, scale) if causal else run_decode(lay, vals, scale)
    G = H_q // H_kv
    qf = W.storage_to_f64(vals.q, lay.geom.dtype)
    cq = lay.cu_q_lens
    for b in range(lay.B):
        K = torch.from_numpy(W.storage_to_f64(W.dense_sequence(lay, vals, b, "k"), W.BF16))
        V = torch.from_numpy(W.storage_to_f64(W.dense_sequence(lay, vals, b, "v"), W.BF16))
        K = K.permute(1, 0, 2).repeat_interleave(G, dim=0)   # [H_q, L, D]
        V = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        n, L = int(lay.q_lens[b]), int(lay.seq_lens[b])
        Q = torch.from_numpy(qf[cq[b]:cq[b + 1]]).permute(1, 0, 2)  # [H_q, n, D]
        qpos = torch.arange(L - n, L).unsqueeze(1)
        kpos = torch.arange(L).unsqueeze(0)
        mask = kpos <= qpos                                          # bottom-right causal
        ref = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
        np.testing.assert_allclose(got[cq[b]:cq[b + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# invariants (ember, "Correctness")
# --------------------------------------------------------------------------
@pytest.mark.parametrize("prefill", [False, True])
def test_block_size_invariance_bit_identical(prefill):
    sl = [1, 17, 64, 100]
    ql = [1, 9, 64, 3] if prefill else None
    outs = []
    base = None
    for P in (1, 2, 3, 7, 16, 64):
        lay = W.custom_layout(8, 2, 64, P, W.BF16, sl, ql, seed=P)
        if base is None:
            base = W.draw_layer_values(lay, np.random.default_rng(7))
        vals = base  # same values by position; only the paging differs
        outs.append(run_prefill(lay, vals, 0.125) if prefill else run_decode(lay, vals, 0.125))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_batch_invariance_bit_identical():
    sl = [40, 3, 77, 12]
    lay = W.custom_layout(8, 4, 128, 16, W.BF16, sl, seed=1)
    vals = W.draw_layer_values(lay, np.random.default_rng(1))
    full = run_decode(lay, vals, 0.09)
    for b in range(lay.B):
        one = W.custom_layout(8, 4, 128, 16, W.BF16, [sl[b]], seed=100 + b)
        cp, cq = lay.cu_prefix, lay.cu_q_lens
        v1 = W.LayerValues(q=vals.q[cq[b]:cq[b + 1]], k_new=vals.k_new[cq[b]:cq[b + 1]],
                           v_new=vals.v_new[cq[b]:cq[b + 1]],
                           k_prefix=vals.k_prefix[cp[b]:cp[b + 1]],
                           v_prefix=vals.v_prefix[cp[b]:cp[b + 1]])
        alone = run_decode(one, v1, 0.09)
        assert np.array_equal(alone[0], full[b])


def test_pool_relabelling_invariance():
    lay = W.custom_layout(4, 2, 64, 4, W.F32, [9, 30, 14], seed=2, spare_blocks=5)
    vals = W.draw_layer_values(lay, np.random.default_rng(4))
    ref = run_decode(lay, vals, 0.2)
    perm = np.random.default_rng(9).permutation(lay.geom.N)
    lay2 = W.Layout(lay.geom, lay.seq_lens, lay.q_lens, perm[lay.block_tables].astype(np.int32),
                    int(perm[lay.spare_block]))
    assert np.array_equal(run_decode(lay2, vals, 0.2), ref)


def test_gqa_equals_mha_with_repeated_kv_heads():
    H_q, H_kv, D = 8, 2, 64
    G = H_q // H_kv
    lay = W.custom_layout(H_q, H_kv, D, 5, W.F32, [12, 29], seed=8)
    vals = W.draw_layer_values(lay, np.random.default_rng(8))
    gqa = run_decode(lay, vals, 0.125)
    lay_m = W.custom_layout(H_q, H_q, D, 5, W.F32, [12, 29], seed=8)
    rep = lambda a: np.repeat(a, G, axis=1)
    vals_m = W.LayerValues(q=vals.q, k_new=rep(vals.k_new), v_new=rep(vals.v_new),
                           k_prefix=rep(vals.k_prefix), v_prefix=rep(vals.v_prefix))
    assert np.array_equal(run_decode(lay_m, vals_m, 0.125), gqa)


def test_prefill_last_row_equals_decode():
    sl, ql = [10, 31, 4], [3, 31, 4]
    lay = W.custom_layout(4, 2, 64, 3, W.BF16, sl, ql, seed=6)
    vals = W.draw_layer_values(lay, np.random.default_rng(6))
    pre = run_prefill(lay, vals, 0.1)
    pools = oracle.build_pools(lay, vals)
    last = lay.cu_q_lens[1:] - 1
    dec = oracle.paged_decode(vals.q[last], pools[0], pools[1], lay.block_tables, lay.seq_lens,
                              0.1, W.BF16, 2)
    assert np.array_equal(pre[last], dec)


# --------------------------------------------------------------------------
# closed forms / special cases
# --------------------------------------------------------------------------
def test_all_keys_equal_gives_mean_of_v():
    lay = W.custom_layout(4, 2, 64, 7, W.F32, [5, 23, 40], [5, 2, 40], seed=4)
    vals = W.draw_layer_values(lay, np.random.default_rng(4))
    vals.k_prefix[:] = vals.k_prefix[:1, :1, :1]   # every key element the same value
    vals.k_new[:] = vals.k_prefix.flat[0]
    out = run_prefill(lay, vals, 0.3)
    G = lay.geom.G
    cq = lay.cu_q_lens
    for b in range(lay.B):
        V = W.dense_sequence(lay, vals, b, "v").astype(np.float64)
        L, n = int(lay.seq_lens[b]), int(lay.q_lens[b])
        for i in range(n):
            vis = L - n + i + 1
            for hq in range(lay.geom.H_q):
                np.testing.assert_allclose(out[cq[b] + i, hq], V[:vis, hq // G].mean(axis=0),
                                           rtol=0, atol=1e-13)


def test_single_position_returns_v0_exactly():
    lay = W.custom_layout(4, 2, 128, 16, W.BF16, [1, 1, 1], seed=9)
    vals = W.draw_layer_values(lay, np.random.default_rng(9))
    out = run_decode(lay, vals, 0.088)
    V = W.storage_to_f64(vals.v_new, W.BF16)
    for hq in range(4):
        assert np.array_equal(out[:, hq], V[:, hq // 2])


def test_zero_query_gives_mean_of_v():
    lay = W.custom_layout(4, 4, 64, 3, W.F32, [8, 19], seed=10)
    vals = W.draw_layer_values(lay, np.random.default_rng(10))
    vals.q[:] = 0
    out = run_decode(lay, vals, 1.0)
    for b in range(lay.B):
        V = W.dense_sequence(lay, vals, b, "v").astype(np.float64)
        np.testing.assert_allclose(out[b], V.mean(axis=0), rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# scatter definition
# --------------------------------------------------------------------------
def test_scatter_skips_negative_slots_and_leaves_other_bytes():
    geom = W.Geometry(H_q=2, H_kv=2, D=64, P=3, N=5, dtype=W.BF16)
    kp = W.empty_pool(geom)
    vp = W.empty_pool(geom)
    before_k = kp.copy()
    rng = np.random.default_rng(0)
    k = W.f32_to_bf16_bits(rng.standard_normal((4, 2, 64), dtype=np.float32))
    v = W.f32_to_bf16_bits(rng.standard_normal((4, 2, 64), dtype=np.float32))
    slots = np.array([7, -1, 0, 14], np.int64)
    oracle.reshape_and_cache(k, v, kp, vp, slots, W.BF16)
    flat_k = kp.reshape(15, 2, 64)
    assert np.array_equal(flat_k[7], k[0]) and np.array_equal(flat_k[0], k[2])
    assert np.array_equal(flat_k[14], k[3])
    untouched = np.ones(15, bool)
    untouched[[7, 0, 14]] = False
    assert np.array_equal(flat_k[untouched], before_k.reshape(15, 2, 64)[untouched])
    assert np.array_equal(vp.reshape(15, 2, 64)[7], v[0])


def test_scatter_rejects_out_of_range_slot():
    geom = W.Geometry(H_q=1, H_kv=1, D=64, P=2, N=2, dtype=W.F32)
    kp = W.empty_pool(geom)
    k = np.zeros((1, 1, 64), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(k, k, kp, kp.copy(), np.array([4], np.int64), W.F32)
    assert np.isnan(kp).all()


def test_decode_rejects_bad_block_id():
    lay = W.custom_layout(2, 1, 64, 4, W.F32, [6], seed=0)
    vals = W.draw_layer_values(lay, np.random.default_rng(0))
    kp, vp = oracle.build_pools(lay, vals)
    bt = lay.block_tables.copy()
    bt[0, 1] = lay.geom.N + 3
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(vals.q, kp, vp, bt, lay.seq_lens, 0.1, W.F32, 1)


def test_oracle_thread_count_does_not_change_results():
    lay = W.custom_layout(8, 2, 64, 16, W.BF16, [50, 3, 90, 17, 33], seed=12)
    vals = W.draw_layer_values(lay, np.random.default_rng(12))
    a = run_decode(lay, vals, 0.125, nthreads=1)
    b = run_decode(lay, vals, 0.125, nthreads=7)
    assert np.array_equal(a, b)


# ---- copy-on-write block copy (tiny-vllm-py "Prefix Sharing") --------------------
def _shared_prefix_pools(step, vals, cow=True):
    """Oracle pools after the shared-prefix step: prefix written once through the
    owner's table, tail blocks copied for the sharers, new tokens scattered."""
    g = step.geom
    kp, vp = W.empty_pool(g), W.empty_pool(g)
    c = step.prefix_len
    oracle.reshape_and_cache(vals.k_prefix[:c], vals.v_prefix[:c], kp, vp, step.prefix_slots, g.dtype)
    if cow:
        oracle.copy_blocks(kp, vp, step.cow_pairs, g.dtype)
    oracle.reshape_and_cache(vals.k_new, vals.v_new, kp, vp, step.post.new_slots(), g.dtype)
    return kp, vp


@pytest.mark.parametrize("prefix_len,P,dtype", [(37, 16, W.F32), (32, 16, W.F32), (5, 4, W.BF16), (70, 7, W.BF16)])
def test_prefix_sharing_with_copy_on_write_matches_brute_force(prefix_len, P, dtype):
    """Requests share prefix blocks; sharers copy the partial tail before appending.
    Decode through the pool equals the contiguous brute force (which never sees a
    pool) for every request, and skipping the copy breaks it."""
    step = W.shared_prefix_step(8, 2, 64, P, dtype, n_req=4, prefix_len=prefix_len, seed=prefix_len)
    vals = W.draw_shared_prefix_values(step, np.random.default_rng(3))
    scale = 1.0 / math.sqrt(64)
    ref = brute_attention(step.post, vals, scale)
    kp, vp = _shared_prefix_pools(step, vals)
    got = oracle.paged_decode(vals.q, kp, vp, step.post.block_tables, step.post.seq_lens, scale, dtype)
    assert np.max(np.abs(got - ref)) <= 1e-12
    if step.cow_pairs.shape[0]:
        kp2, vp2 = _shared_prefix_pools(step, vals, cow=False)
        bad = oracle.paged_decode(vals.q, kp2, vp2, step.post.block_tables, step.post.seq_lens, scale, dtype)
        assert not np.allclose(bad[1:], ref[1:], equal_nan=False)   # sharers read unwritten (NaN) rows
        np.testing.assert_allclose(bad[0], ref[0], rtol=0, atol=1e-12)  # the owner kept the original


def test_copy_blocks_leaves_sources_and_other_blocks_and_reads_before_writing():
    """Sources and blocks no pair names keep their bytes; a block that is copied
    and also copied from (src of one pair, dst of another) is read before it is
    overwritten."""
    g = W.Geometry(H_q=4, H_kv=2, D=64, P=4, N=6, dtype=W.BF16)
    rng = np.random.default_rng(5)
    kp = W._draw(rng, (g.N, g.P, g.H_kv, g.D), g.dtype, 1.0)
    vp = W._draw(rng, (g.N, g.P, g.H_kv, g.D), g.dtype, 1.0)
    k0, v0 = kp.copy(), vp.copy()
    oracle.copy_blocks(kp, vp, np.array([[1, 4], [4, 2]], np.int32), g.dtype)   # 4 <- 1, 2 <- old 4
    assert np.array_equal(kp[4], k0[1]) and np.array_equal(vp[4], v0[1])
    assert np.array_equal(kp[2], k0[4]) and np.array_equal(vp[2], v0[4])
    for blk in (0, 1, 3, 5):
        assert np.array_equal(kp[blk], k0[blk]) and np.array_equal(vp[blk], v0[blk])


def test_copy_blocks_on_fp8_code_pools_moves_whole_blocks_of_bytes():
    """e4m3 code pools (one byte an element): the same block copy, byte for byte."""
    rng = np.random.default_rng(6)
    kp = rng.integers(0, 256, (5, 16, 8, 128), dtype=np.uint8)
    vp = rng.integers(0, 256, (5, 16, 8, 128), dtype=np.uint8)
    k0, v0 = kp.copy(), vp.copy()
    oracle.copy_blocks(kp, vp, np.array([[3, 0], [0, 4]], np.int32), "fp8")   # 0 <- 3, 4 <- old 0
    assert np.array_equal(kp[0], k0[3]) and np.array_equal(vp[0], v0[3])
    assert np.array_equal(kp[4], k0[0]) and np.array_equal(vp[4], v0[0])
    for blk in (1, 2, 3):
        assert np.array_equal(kp[blk], k0[blk]) and np.array_equal(vp[blk], v0[blk])


def test_copy_blocks_rejects_out_of_range_ids_before_writing():
    g = W.Geometry(H_q=4, H_kv=2, D=64, P=4, N=3, dtype=W.F32)
    kp, vp = W.empty_pool(g), W.empty_pool(g)
    k0 = kp.copy()
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(kp, vp, np.array([[0, 1], [0, 3]], np.int32), g.dtype)
    assert np.array_equal(kp.view(np.uint32), k0.view(np.uint32))


# ---- fp8 e4m3 KV pools (ember "Deliberately out of scope": paged KV quantization) ----
def _torch():
    return pytest.importorskip("torch")


def test_e4m3_decode_matches_torch_float8_e4m3fn_for_all_codes():
    torch = _torch()
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().double().numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rounding_in_range_and_saturates_beyond():
    torch = _torch()
    rng = np.random.default_rng(7)
    finite = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = (finite[1:] + finite[:-1]) / 2                       # exact ties
    ys = np.concatenate([rng.uniform(-464, 464, 4000), rng.standard_normal(2000) * 0.01, mids, -mids,
                         finite, -finite, [0.0, -0.0, 2.0 ** -10, 2.0 ** -11]]).astype(np.float32)
    ref = torch.from_numpy(ys).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(y)) for y in ys], np.uint8)
    assert np.array_equal(got, ref)
    for y, code in [(500.0, 0x7E), (-1e9, 0xFE), (float("inf"), 0x7E), (448.0, 0x7E)]:
        assert oracle.e4m3_encode(y) == code
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def _fp8_case(seed=0, k_scale=0.0625, v_scale=0.25):
    lay = W.custom_layout(8, 2, 64, 16, W.BF16, [40, 17, 64, 1], seed=seed)
    vals = W.draw_layer_values(lay, np.random.default_rng(seed + 1))
    g = lay.geom
    shape = (g.N, g.P, g.H_kv, g.D)
    kp, vp = np.full(shape, 0x7F, np.uint8), np.full(shape, 0x7F, np.uint8)   # NaN codes everywhere
    oracle.reshape_and_cache_fp8(vals.k_prefix, vals.v_prefix, kp, vp, lay.prefix_slots(), k_scale, v_scale)
    oracle.reshape_and_cache_fp8(vals.k_new, vals.v_new, kp, vp, lay.new_slots(), k_scale, v_scale)
    return lay, vals, kp, vp


def test_fp8_scatter_codes_match_torch_quantization():
    """code = e4m3(float(x) * float32(1/scale)), checked against torch's float8 cast."""
    torch = _torch()
    k_scale, v_scale = 0.0625, 0.3
    lay, vals, kp, vp = _fp8_case(k_scale=k_scale, v_scale=v_scale)
    for rows, slots in ((vals.k_new, lay.new_slots()), (vals.k_prefix, lay.prefix_slots())):
        x = torch.from_numpy(W.bf16_bits_to_f32(rows))
        want = (x * torch.tensor(np.float32(1.0) / np.float32(k_scale))).to(torch.float8_e4m3fn).view(torch.uint8)
        got = kp.reshape(-1, lay.geom.H_kv, lay.geom.D)[slots]
        assert np.array_equal(got, want.numpy())
    x = torch.from_numpy(W.bf16_bits_to_f32(vals.v_new))
    want = (x * torch.tensor(np.float32(1.0) / np.float32(v_scale))).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(vp.reshape(-1, lay.geom.H_kv, lay.geom.D)[lay.new_slots()], want.numpy())


def test_fp8_decode_matches_brute_force_on_dequantized_values():
    """Decode over e4m3 pools equals the contiguous brute force on the dequantized
    sequences (scale * value of each code, quantized here by torch), and swapping
    the K and V scales breaks it."""
    torch = _torch()
    k_scale, v_scale = 0.0625, 0.25
    lay, vals, kp, vp = _fp8_case(k_scale=k_scale, v_scale=v_scale)
    g = lay.geom
    scale = 1.0 / math.sqrt(g.D)
    got = oracle.paged_decode_fp8(vals.q, kp, vp, lay.block_tables, lay.seq_lens, scale, k_scale, v_scale)

    def deq(rows, s):
        x = torch.from_numpy(W.bf16_bits_to_f32(rows))
        c = (x * torch.tensor(np.float32(1.0) / np.float32(s))).to(torch.float8_e4m3fn)
        return c.double().numpy() * s

    q = W.storage_to_f64(vals.q, g.dtype)
    cp, cq = lay.cu_prefix, lay.cu_q_lens
    ref = np.zeros_like(got)
    for b in range(lay.B):
        K = np.concatenate([deq(vals.k_prefix[cp[b]:cp[b + 1]], k_scale), deq(vals.k_new[cq[b]:cq[b + 1]], k_scale)])
        V = np.concatenate([deq(vals.v_prefix[cp[b]:cp[b + 1]], v_scale), deq(vals.v_new[cq[b]:cq[b + 1]], v_scale)])
        for hq in range(g.H_q):
            s = scale * (K[:, hq // g.G, :] @ q[b, hq])
            w = np.exp(s - s.max())
            ref[b, hq] = (w @ V[:, hq // g.G, :]) / w.sum()
    assert np.max(np.abs(got - ref)) <= 1e-12
    swapped = oracle.paged_decode_fp8(vals.q, kp, vp, lay.block_tables, lay.seq_lens, scale, v_scale, k_scale)
    assert np.max(np.abs(swapped - ref)) > 1e-3


def _deq_per_head(torch, rows, scales):
    """rows [T, H_kv, D] bf16 bits -> scale_h * e4m3(float32(x) * float32(1/scale_h)), by torch."""
    x = torch.from_numpy(W.bf16_bits_to_f32(rows))
    inv = torch.tensor((np.float32(1.0) / np.asarray(scales, np.float32)).astype(np.float32)).view(1, -1, 1)
    c = (x * inv).to(torch.float8_e4m3fn)
    # the scales are float32 numbers (the pool descriptor's type), widened exactly
    return c, c.double().numpy() * np.asarray(scales, np.float32).astype(np.float64).reshape(1, -1, 1)


def test_fp8_per_head_scales_scatter_and_decode():
    """One scale per KV head (the per-head variant of the fp8 pool): head h's
    codes are torch's e4m3 cast of x * float32(1/scale_h), decode equals the
    contiguous brute force on the per-head dequantized values, equal per-head scales
    reproduce the per-tensor result exactly, and swapping two heads' scales breaks it."""
    torch = _torch()
    ks, vs = [0.0625, 0.3], [0.25, 0.011]
    lay, vals, kp, vp = _fp8_case(k_scale=ks, v_scale=vs)
    g = lay.geom
    for rows, slots, pool, sc in ((vals.k_new, lay.new_slots(), kp, ks), (vals.v_prefix, lay.prefix_slots(), vp, vs)):
        want, _ = _deq_per_head(torch, rows, sc)
        assert np.array_equal(pool.reshape(-1, g.H_kv, g.D)[slots], want.view(torch.uint8).numpy())
    scale = 1.0 / math.sqrt(g.D)
    got = oracle.paged_decode_fp8(vals.q, kp, vp, lay.block_tables, lay.seq_lens, scale, ks, vs)
    q = W.storage_to_f64(vals.q, g.dtype)
    cp, cq = lay.cu_prefix, lay.cu_q_lens
    ref = np.zeros_like(got)
    for b in range(lay.B):
        K = np.concatenate([_deq_per_head(torch, vals.k_prefix[cp[b]:cp[b + 1]], ks)[1],
                            _deq_per_head(torch, vals.k_new[cq[b]:cq[b + 1]], ks)[1]])
        V = np.concatenate([_deq_per_head(torch, vals.v_prefix[cp[b]:cp[b + 1]], vs)[1],
                            _deq_per_head(torch, vals.v_new[cq[b]:cq[b + 1]], vs)[1]])
        for hq in range(g.H_q):
            s = scale * (K[:, hq // g.G, :] @ q[b, hq])
            w = np.exp(s - s.max())
            ref[b, hq] = (w @ V[:, hq // g.G, :]) / w.sum()
    assert np.max(np.abs(got - ref)) <= 1e-12
    swapped = oracle.paged_decode_fp8(vals.q, kp, vp, lay.block_tables, lay.seq_lens, scale, ks[::-1], vs)
    assert np.max(np.abs(swapped - ref)) > 1e-3
    # equal per-head scales are the per-tensor pool, byte for byte and output for output
    lay1, vals1, kp1, vp1 = _fp8_case(k_scale=0.0625, v_scale=0.25)
    lay2, vals2, kp2, vp2 = _fp8_case(k_scale=[0.0625, 0.0625], v_scale=[0.25, 0.25])
    assert np.array_equal(kp1, kp2) and np.array_equal(vp1, vp2)
    a = oracle.paged_decode_fp8(vals1.q, kp1, vp1, lay1.block_tables, lay1.seq_lens, scale, 0.0625, 0.25)
    c = oracle.paged_decode_fp8(vals2.q, kp2, vp2, lay2.block_tables, lay2.seq_lens, scale, [0.0625] * 2, [0.25] * 2)
    assert np.array_equal(a, c)

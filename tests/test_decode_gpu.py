"""wf_paged_decode on the GPU against the fp64 oracle.

Pools are NaN everywhere no live position lives (unused table entries point at a
NaN block), so any read past seq_len or of a stale block shows up as NaN.
Tolerances: fp32 KV max abs <= 1e-4; bf16 KV max abs <= 2e-2 and mean abs <= 2e-3.
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
    "tiny_f32": lambda: W.tiny_decode(0),
    "gpt2_bf16": lambda: W.gpt2_decode(0),
    "llama1b_bf16": lambda: W.llama1b_decode(0),
    "gqa3_P1": lambda: W.custom_layout(6, 2, 64, 1, W.BF16, [1, 2, 130, 257], seed=1),
    "gqa8_P7_f32": lambda: W.custom_layout(16, 2, 128, 7, W.F32, [300, 1, 129, 128, 127], seed=2),
    "gqa2_P3_f32": lambda: W.custom_layout(4, 2, 64, 3, W.F32, [17, 64, 65, 2], seed=3),
    "long_P64": lambda: W.custom_layout(8, 4, 128, 64, W.BF16, [5000, 33, 128, 129], seed=4),
    "mha12_two_head_groups": lambda: W.custom_layout(12, 12, 64, 16, W.BF16, [700, 1, 256], seed=5),
    "mha_f32_D128": lambda: W.custom_layout(4, 4, 128, 16, W.F32, [1000, 31], seed=6),
    "gqa4_D128_ragged": lambda: W.custom_layout(32, 8, 128, 16, W.BF16,
                                                [1, 15, 16, 17, 127, 128, 129, 255, 256, 2049], seed=7),
    # tensor-core decode at D = 64 (P.V over a zero upper half of V^T)
    "gqa4_D64_ragged": lambda: W.custom_layout(32, 8, 64, 16, W.BF16,
                                               [1, 15, 16, 17, 127, 128, 129, 255, 256, 2049], seed=14),
    "gqa2_D64_P32_long": lambda: W.custom_layout(16, 8, 64, 32, W.BF16, [4000, 1, 300, 64, 33], seed=15),
    # around the work-item boundaries: 256 positions (tensor cores, D = 128) and 64
    # positions (CUDA-core kernel)
    "gqa4_D128_items256": lambda: W.custom_layout(32, 8, 128, 16, W.BF16,
                                                  [255, 256, 257, 511, 512, 513, 768, 769], seed=16),
    "mha12_items64": lambda: W.custom_layout(12, 12, 64, 16, W.BF16, [63, 64, 65, 128, 129, 193], seed=17),
    # tensor-core decode, group of 2 at D = 128 (H_q = 16, H_kv = 8)
    "gqa2_D128_ragged": lambda: W.custom_layout(16, 8, 128, 16, W.BF16,
                                                [1, 15, 16, 17, 255, 256, 257, 1000, 3001], seed=18),
    # tensor-core decode at D = 128 with blocks of 32 and 64 positions (a 16-position
    # tile is a sub-range of one block)
    "gqa4_D128_P32": lambda: W.custom_layout(32, 8, 128, 32, W.BF16, [1, 31, 32, 33, 300, 2049], seed=19),
    "gqa4_D128_P64": lambda: W.custom_layout(32, 8, 128, 64, W.BF16, [1, 63, 64, 65, 700, 1500], seed=20),
    "gqa2_D128_P64": lambda: W.custom_layout(16, 8, 128, 64, W.BF16, [2, 64, 129, 513, 1200], seed=21),
    # tensor-core decode for other KV-head counts: a tile holds 8 / HT boxes of 16
    # positions of HT heads (HT = the largest power of two <= 8 dividing H_kv)
    "mha8_D128": lambda: W.custom_layout(8, 8, 128, 16, W.BF16, [1, 17, 255, 256, 257, 900], seed=22),
    "mha16_D64_two_groups": lambda: W.custom_layout(16, 16, 64, 16, W.BF16, [5, 128, 129, 1000], seed=23),
    "gqa2_kv16_D128": lambda: W.custom_layout(32, 16, 128, 32, W.BF16, [3, 300, 1100], seed=24),
    "gqa4_kv2_D128": lambda: W.custom_layout(8, 2, 128, 16, W.BF16, [1, 16, 17, 63, 64, 65, 700, 2000], seed=25),
    "gqa2_kv6_D64_P32": lambda: W.custom_layout(12, 6, 64, 32, W.BF16, [1, 31, 33, 128, 129, 640], seed=26),
    "mqa_gqa4_kv1_D128": lambda: W.custom_layout(4, 1, 128, 16, W.BF16, [1, 15, 16, 17, 127, 128, 129, 1500], seed=27),
    "mqa_kv1_D64": lambda: W.custom_layout(1, 1, 64, 16, W.BF16, [2, 100, 129, 700], seed=28),
    "gqa2_kv3_D64": lambda: W.custom_layout(6, 3, 64, 16, W.BF16, [1, 44, 128, 300, 1024], seed=29),
    "gqa4_kv4_D64_P64": lambda: W.custom_layout(16, 4, 64, 64, W.BF16, [64, 65, 128, 129, 1000], seed=30),
    # a group of 8 stays on the CUDA cores
    "gqa8_bf16_cuda_cores": lambda: W.custom_layout(16, 2, 128, 16, W.BF16, [1, 300, 1029], seed=31),
    # large blocks, up to the largest block size the calls accept (1024 positions)
    "gqa4_D128_P256": lambda: W.custom_layout(32, 8, 128, 256, W.BF16, [1, 255, 256, 257, 1000, 3001], seed=32),
    "gqa2_D64_P1024": lambda: W.custom_layout(16, 8, 64, 1024, W.BF16, [1, 1023, 1024, 1025, 2500], seed=33),
}


def _oracle_decode(lay, vals, scale):
    kp, vp = oracle.build_pools(lay, vals)
    return oracle.paged_decode(vals.q, kp, vp, lay.block_tables, lay.seq_lens, scale, lay.geom.dtype)


@pytest.mark.parametrize("name", list(CASES.keys()))
def test_decode_matches_oracle(name):
    lay = CASES[name]()
    vals = W.draw_layer_values(lay, np.random.default_rng(31))
    scale = G.default_scale(lay.geom.D)
    st = G.dev_status()
    pools = G.build_dev_pools(lay, vals, st)
    out = G.run_decode(lay, vals, pools, scale, st)
    got = G.from_dev(out, lay.geom.dtype)
    ref = _oracle_decode(lay, vals, scale)
    G.assert_close(got, ref, lay.geom.dtype, name)
    assert wf.wf_device_status_fetch(st) == 0


def test_decode_block_size_invariance():
    """The same values by position, paged with P in {1, 2, 3, 7, 16, 32, 64}.

    Llama-3-8B heads (H_q 32, H_kv 8, D 128, bf16): block sizes that are multiples of
    16 run the tensor-core kernel, the others the CUDA-core kernel.  Every P is
    compared with the oracle, and within each kernel the output bytes are identical
    for every P: the tile order depends only on the logical position."""
    sl = [1, 17, 130, 300, 1025]
    outs = {}
    base = None
    ref = None
    for P in (1, 2, 3, 7, 16, 32, 64):
        lay = W.custom_layout(32, 8, 128, P, W.BF16, sl, seed=P)
        want = wf.WF_KERNEL_TENSOR_CORES if P % 16 == 0 else wf.WF_KERNEL_CUDA_CORES
        assert G.decode_kernel(lay.geom) == want, P
        if base is None:
            base = W.draw_layer_values(lay, np.random.default_rng(8))
            ref = _oracle_decode(lay, base, 0.088)
        st = G.dev_status()
        pools = G.build_dev_pools(lay, base, st)
        outs[P] = G.run_decode(lay, base, pools, 0.088, st)
        assert wf.wf_device_status_fetch(st) == 0
        G.assert_close(G.from_dev(outs[P], W.BF16), ref, W.BF16, f"P={P}")
    for fam in ((1, 2, 3, 7), (16, 32, 64)):
        first = G.storage_bytes(outs[fam[0]])
        for P in fam[1:]:
            assert np.array_equal(G.storage_bytes(outs[P]), first), P


def test_decode_batch_invariance_bit_identical():
    """A sequence decoded alone gives the same bytes as inside a batch."""
    torch = G.torch_mod()
    lay = W.custom_layout(32, 8, 128, 16, W.BF16, [3000, 5, 129, 640], seed=9)
    vals = W.draw_layer_values(lay, np.random.default_rng(9))
    kp, vp = G.build_dev_pools(lay, vals)
    full = G.storage_bytes(G.run_decode(lay, vals, (kp, vp), 0.088)).reshape(lay.B, -1)
    for b in range(lay.B):
        one = W.Layout(lay.geom, lay.seq_lens[b:b + 1].copy(), lay.q_lens[b:b + 1].copy(),
                       lay.block_tables[b:b + 1].copy(), lay.spare_block)
        v1 = W.LayerValues(q=vals.q[b:b + 1], k_new=vals.k_new[b:b + 1], v_new=vals.v_new[b:b + 1],
                           k_prefix=vals.k_prefix[:0], v_prefix=vals.v_prefix[:0])
        alone = G.storage_bytes(G.run_decode(one, v1, (kp, vp), 0.088, max_seq_len=lay.M * lay.geom.P))
        assert np.array_equal(alone, full[b])


def _subpool(kp, vp, lay, seqs):
    """Host copies of just the blocks the chosen sequences use, with remapped tables."""
    torch = G.torch_mod()
    P = lay.geom.P
    nb = [-(-int(lay.seq_lens[b]) // P) for b in seqs]
    used = np.unique(np.concatenate([lay.block_tables[b, :n] for b, n in zip(seqs, nb)]))
    remap = {int(x): i for i, x in enumerate(used)}
    idx = torch.from_numpy(used.astype(np.int64)).cuda()
    hk = kp.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    hv = vp.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    M = max(nb)
    bt = np.zeros((len(seqs), M), np.int32)
    for i, (b, n) in enumerate(zip(seqs, nb)):
        bt[i, :n] = [remap[int(x)] for x in lay.block_tables[b, :n]]
    return hk, hv, bt


@pytest.mark.parametrize("B", [118, 231])
def test_decode_llama8b_full_size_sampled(B):
    """Full Llama-3-8B-shaped batch on the device (one layer, launch exactly as the
    benchmark does); the oracle recomputes a sample of sequences one by one."""
    torch = G.torch_mod()
    lay = W.llama8b_decode(B, seed=0)
    g = lay.geom
    kp, vp = W.device_pools(lay, seed=11)
    q, k_new, v_new = W.device_step_values(lay, seed=12)
    order = np.argsort(lay.seq_lens)
    seqs = sorted(set(order[:4].tolist() + order[-4:].tolist() + order[:: max(1, B // 12)].tolist()))
    # oracle inputs: host copies taken BEFORE the GPU writes this step's tokens
    hk, hv, hbt = _subpool(kp, vp, lay, seqs)
    new_slots = lay.new_slots()
    st = G.dev_status()
    wf.wf_reshape_and_cache(k_new, v_new, kp, vp, torch.from_numpy(new_slots).cuda(), st)
    out = torch.empty_like(q)
    ws = torch.empty(wf.wf_paged_decode_workspace_size(B, g.H_q, lay.max_seq_len, wf.pool_desc(kp)),
                     dtype=torch.uint8, device="cuda")
    wf.wf_paged_decode(out, q, kp, vp, torch.from_numpy(lay.block_tables).cuda(),
                       torch.from_numpy(lay.seq_lens).cuda(), lay.max_seq_len, 1 / math.sqrt(g.D), ws, st)
    assert wf.wf_device_status_fetch(st) == 0
    # oracle: its own scatter of the sampled sequences' new rows, then decode
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    hq, hkn, hvn = bits(q[seqs]), bits(k_new[seqs]), bits(v_new[seqs])
    sub = W.Layout(W.Geometry(g.H_q, g.H_kv, g.D, g.P, hk.shape[0], g.dtype), lay.seq_lens[seqs],
                   np.ones(len(seqs), np.int32), hbt, 0)
    oracle.reshape_and_cache(hkn, hvn, hk, hv, sub.new_slots(), g.dtype)
    ref = oracle.paged_decode(hq, hk, hv, hbt, lay.seq_lens[seqs], 1 / math.sqrt(g.D), g.dtype)
    got = G.from_dev(out[seqs], g.dtype)
    G.assert_close(got, ref, g.dtype, f"llama8b B={B}")
    # every output of the batch is finite (no NaN-poisoned slot was read)
    assert torch.isfinite(out.float()).all()


def test_decode_flags_bad_seq_len_and_bad_block():
    torch = G.torch_mod()
    lay = W.custom_layout(8, 2, 64, 16, W.BF16, [40, 50, 60], seed=10)
    vals = W.draw_layer_values(lay, np.random.default_rng(10))
    kp, vp = G.build_dev_pools(lay, vals)
    ref = _oracle_decode(lay, vals, 0.125)
    # sequence 1 claims more tokens than max_seq_len: skipped and flagged
    bad = W.Layout(lay.geom, np.array([40, 999, 60], np.int32), lay.q_lens, lay.block_tables,
                   lay.spare_block)
    st = G.dev_status()
    out = G.run_decode(bad, vals, (kp, vp), 0.125, st, max_seq_len=64)
    assert wf.wf_device_status_fetch(st) == wf.WF_DEV_BAD_SEQLEN
    got = G.from_dev(out, W.BF16)
    G.assert_close(got[[0, 2]], ref[[0, 2]], W.BF16, "untouched sequences")
    # a block id past N in sequence 2's table: its rows are skipped and flagged
    bt = lay.block_tables.copy()
    bt[2, 1] = lay.geom.N + 7
    bad2 = W.Layout(lay.geom, lay.seq_lens, lay.q_lens, bt, lay.spare_block)
    st2 = G.dev_status()
    G.run_decode(bad2, vals, (kp, vp), 0.125, st2)
    assert wf.wf_device_status_fetch(st2) & wf.WF_DEV_BAD_BLOCK


def test_decode_empty_batch_is_a_no_op():
    torch = G.torch_mod()
    g = W.Geometry(H_q=4, H_kv=2, D=64, P=16, N=4, dtype=W.BF16)
    kp = G.empty_dev_pool(g)
    q = torch.empty((0, 4, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    bt = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    sl = torch.zeros(0, dtype=torch.int32, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    wf.wf_paged_decode(out, q, kp, kp.clone(), bt, sl, 16, 0.125, ws)


@pytest.mark.parametrize("H_q,H_kv,D,P", [(32, 8, 128, 16), (8, 2, 64, 16)])
def test_decode_workspace_left_dirty_is_fine_and_reusable(H_q, H_kv, D, P):
    """The workspace needs no initialisation: filled with 0xFF bytes, then reused by
    a second call, it gives the same bytes both times, within tolerance of the oracle
    (the tensor-core kernels keep their work-item queue in it)."""
    torch = G.torch_mod()
    lay = W.custom_layout(H_q, H_kv, D, P, W.BF16, [3000, 5, 129, 640, 1, 2048], seed=12)
    vals = W.draw_layer_values(lay, np.random.default_rng(12))
    kp, vp = G.build_dev_pools(lay, vals)
    q = G.to_dev(vals.q, W.BF16)
    ws = torch.full((wf.wf_paged_decode_workspace_size(lay.B, H_q, lay.max_seq_len, wf.pool_desc(kp)),), 255,
                    dtype=torch.uint8, device="cuda")
    bt, sl = torch.from_numpy(lay.block_tables).cuda(), torch.from_numpy(lay.seq_lens).cuda()
    outs = []
    for _ in range(2):
        out = torch.empty_like(q)
        st = G.dev_status()
        wf.wf_paged_decode(out, q, kp, vp, bt, sl, lay.max_seq_len, 0.088, ws, st)
        assert wf.wf_device_status_fetch(st) == 0
        outs.append(G.storage_bytes(out))
    assert np.array_equal(outs[0], outs[1])
    G.assert_close(G.from_dev(out, W.BF16), _oracle_decode(lay, vals, 0.088), W.BF16, "dirty workspace")


def test_decode_tensor_core_path_flags_bad_seq_len():
    """Llama-3-8B heads (tensor-core kernel): a sequence longer than max_seq_len is
    skipped and flagged; the others are decoded as usual."""
    lay = W.custom_layout(32, 8, 128, 16, W.BF16, [40, 50, 300, 60], seed=13)
    vals = W.draw_layer_values(lay, np.random.default_rng(13))
    kp, vp = G.build_dev_pools(lay, vals)
    ref = _oracle_decode(lay, vals, 0.088)
    bad = W.Layout(lay.geom, np.array([40, 50, 9999, 60], np.int32), lay.q_lens, lay.block_tables,
                   lay.spare_block)
    st = G.dev_status()
    out = G.run_decode(bad, vals, (kp, vp), 0.088, st, max_seq_len=lay.max_seq_len)
    assert wf.wf_device_status_fetch(st) == wf.WF_DEV_BAD_SEQLEN
    got = G.from_dev(out, W.BF16)
    G.assert_close(got[[0, 1, 3]], ref[[0, 1, 3]], W.BF16, "untouched sequences")

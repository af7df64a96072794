"""fp8 e4m3 KV pools on the GPU: the quantizing scatter bit-exact against the
oracle's codes, and paged decode over code pools within the bf16 tolerance of the
oracle's fp64 decode of the dequantized values (ember, "Deliberately out of
scope": paged KV quantization).

Pools start as the e4m3 NaN code (0x7F) everywhere, so a decode that reads a slot
no live position owns shows up as NaN.
"""
import math

import numpy as np
import pytest

import oracle
from paged_kv_cache_wf_gb300 import binding as wf
from paged_kv_cache_wf_gb300 import workloads as W
from tests import _gpu as G

pytestmark = pytest.mark.gpu

NAN_CODE = 0x7F


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = G.torch_mod()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_cache_wf_gb300 import build
    build.build()


def _empty_codes(g):
    return np.full((g.N, g.P, g.H_kv, g.D), NAN_CODE, np.uint8)


def _dev_u8(a):
    torch = G.torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda()


def _pools_both(lay, vals, ks, vs, status=None):
    """The same scatters (prefix rows, then this step's rows) on the GPU and in the oracle."""
    torch = G.torch_mod()
    g = lay.geom
    hk, hv = _empty_codes(g), _empty_codes(g)
    dk, dv = _dev_u8(hk), _dev_u8(hv)
    for k, v, s in ((vals.k_prefix, vals.v_prefix, lay.prefix_slots()), (vals.k_new, vals.v_new, lay.new_slots())):
        if k.shape[0] == 0:
            continue
        wf.wf_reshape_and_cache(G.to_dev(k, W.BF16), G.to_dev(v, W.BF16), dk, dv, torch.from_numpy(s).cuda(),
                                status, k_scale=ks, v_scale=vs)
        oracle.reshape_and_cache_fp8(k, v, hk, hv, s, ks, vs)
    return (dk, dv), (hk, hv)


@pytest.mark.parametrize("H_kv,D,P,T,ks,vs", [
    (8, 128, 16, 300, 1 / 64, 1 / 96),      # Llama-3-8B row; 1/96 is not a power of two
    (2, 64, 3, 77, 0.37, 2.5e-3),           # odd block size; small v_scale saturates many codes
    (12, 64, 1, 40, 1.0, 1.0),              # one-slot blocks, unit scales (subnormal codes)
])
def test_fp8_scatter_bit_exact(H_kv, D, P, T, ks, vs):
    torch = G.torch_mod()
    N = -(-T // P) + 3
    rng = np.random.default_rng(T)
    x = rng.standard_normal((2, T, H_kv, D)).astype(np.float32)
    x[:, ::5] *= 300.0                       # some rows well past +-448 * scale: saturation
    x[:, 1::7] *= 1e-3                       # and some deep in the subnormal codes
    x[0, 2, 0, :4] = [0.0, -0.0, 448.0 * ks, -449.0 * ks]
    k, v = W.f32_to_bf16_bits(x[0]), W.f32_to_bf16_bits(x[1])
    slots = rng.permutation(N * P)[:T].astype(np.int64)
    slots[3] = -1                            # padding token: nothing written
    g = W.Geometry(H_q=H_kv, H_kv=H_kv, D=D, P=P, N=N, dtype=W.BF16)
    hk, hv = _empty_codes(g), _empty_codes(g)
    dk, dv = _dev_u8(hk), _dev_u8(hv)
    st = G.dev_status()
    wf.wf_reshape_and_cache(G.to_dev(k, W.BF16), G.to_dev(v, W.BF16), dk, dv, torch.from_numpy(slots).cuda(), st,
                            k_scale=ks, v_scale=vs)
    oracle.reshape_and_cache_fp8(k, v, hk, hv, slots, ks, vs)
    assert np.array_equal(dk.cpu().numpy(), hk)
    assert np.array_equal(dv.cpu().numpy(), hv)
    assert wf.wf_device_status_fetch(st) == 0
    # the case exercises what it says: saturated codes, subnormal codes, both zeros
    assert ((hv & 0x7F) == 0x7E).any() and ((hk & 0x78) == 0).any()


def test_fp8_scatter_flags_bad_slot_and_writes_the_rest():
    torch = G.torch_mod()
    g = W.Geometry(H_q=2, H_kv=2, D=64, P=4, N=6, dtype=W.BF16)
    rng = np.random.default_rng(3)
    k = W._draw(rng, (5, 2, 64), W.BF16, 1.0)
    v = W._draw(rng, (5, 2, 64), W.BF16, 1.0)
    slots = np.array([0, 24, 5, 1 << 40, 23], np.int64)      # 24 and 2^40 are outside N*P
    hk, hv = _empty_codes(g), _empty_codes(g)
    dk, dv = _dev_u8(hk), _dev_u8(hv)
    st = G.dev_status()
    wf.wf_reshape_and_cache(G.to_dev(k, W.BF16), G.to_dev(v, W.BF16), dk, dv, torch.from_numpy(slots).cuda(), st,
                            k_scale=0.05, v_scale=0.05)
    keep = [0, 2, 4]
    oracle.reshape_and_cache_fp8(k[keep], v[keep], hk, hv, slots[keep], 0.05, 0.05)
    assert np.array_equal(dk.cpu().numpy(), hk) and np.array_equal(dv.cpu().numpy(), hv)
    assert wf.wf_device_status_fetch(st) == wf.WF_DEV_BAD_SLOT


CASES = {
    # Llama-3-8B heads (G=4), ragged lengths around the 16-position tile
    "gqa4_ragged": lambda: W.custom_layout(32, 8, 128, 16, W.BF16,
                                           [1, 15, 16, 17, 127, 128, 129, 255, 256, 2049], seed=21),
    # G=2, larger blocks
    "gqa2_P32": lambda: W.custom_layout(16, 8, 128, 32, W.BF16, [1, 300, 1000, 64, 33], seed=22),
    # around the 256-position work items
    "gqa4_items256": lambda: W.custom_layout(32, 8, 128, 16, W.BF16, [255, 256, 257, 511, 512, 513, 1025], seed=24),
    # shapes the tensor-core kernel does not take: the CUDA-core kernel widens the codes
    "core_mha12_D64": lambda: W.custom_layout(12, 12, 64, 16, W.BF16, [700, 1, 256, 63, 65], seed=25),
    "core_gqa8_D128_P7": lambda: W.custom_layout(16, 2, 128, 7, W.BF16, [300, 1, 129, 128, 127], seed=26),
    # D = 64: two 16-position sub-tiles of 64-byte code rows per stage
    "gqa4_D64": lambda: W.custom_layout(32, 8, 64, 16, W.BF16, [1, 15, 16, 17, 31, 32, 33, 257, 2049], seed=27),
    "gqa2_D64_P32": lambda: W.custom_layout(16, 8, 64, 32, W.BF16, [2, 33, 64, 300, 1000], seed=32),
    # one long context in 64-slot blocks (many splits: combine path)
    "gqa4_long_P64": lambda: W.custom_layout(32, 8, 128, 64, W.BF16, [5000, 33, 128], seed=23),
}


@pytest.mark.parametrize("name", list(CASES.keys()))
@pytest.mark.parametrize("ks,vs", [(1 / 64, 1 / 96), (0.011, 0.5)])
def test_fp8_decode_matches_oracle(name, ks, vs):
    torch = G.torch_mod()
    lay = CASES[name]()
    vals = W.draw_layer_values(lay, np.random.default_rng(41))
    g = lay.geom
    scale = G.default_scale(g.D)
    st = G.dev_status()
    (dk, dv), (hk, hv) = _pools_both(lay, vals, ks, vs, st)
    assert np.array_equal(dk.cpu().numpy(), hk) and np.array_equal(dv.cpu().numpy(), hv)
    q = G.to_dev(vals.q, W.BF16)
    out = torch.empty_like(q)
    ws = torch.empty(wf.wf_paged_decode_workspace_size(lay.B, g.H_q, lay.max_seq_len, wf.pool_desc(dk, ks, vs)),
                     dtype=torch.uint8, device="cuda")
    wf.wf_paged_decode(out, q, dk, dv, torch.from_numpy(lay.block_tables).cuda(),
                       torch.from_numpy(lay.seq_lens).cuda(), lay.max_seq_len, scale, ws, st, k_scale=ks, v_scale=vs)
    assert wf.wf_device_status_fetch(st) == 0
    ref = oracle.paged_decode_fp8(vals.q, hk, hv, lay.block_tables, lay.seq_lens, scale, ks, vs)
    G.assert_close(G.from_dev(out, W.BF16), ref, W.BF16, f"fp8 {name}")


def test_fp8_decode_batch_invariance_bit_identical():
    """A sequence decoded alone gives the same bytes as inside a batch."""
    torch = G.torch_mod()
    lay = W.custom_layout(32, 8, 128, 16, W.BF16, [3000, 5, 129, 640], seed=29)
    vals = W.draw_layer_values(lay, np.random.default_rng(29))
    (dk, dv), _ = _pools_both(lay, vals, 1 / 64, 1 / 64)
    g = lay.geom

    def run(b_idx, msl):
        q = G.to_dev(vals.q[b_idx], W.BF16)
        out = torch.empty_like(q)
        ws = torch.empty(wf.wf_paged_decode_workspace_size(len(b_idx), g.H_q, msl, wf.pool_desc(dk, 1 / 64, 1 / 64)),
                         dtype=torch.uint8, device="cuda")
        wf.wf_paged_decode(out, q, dk, dv, torch.from_numpy(np.ascontiguousarray(lay.block_tables[b_idx])).cuda(),
                           torch.from_numpy(np.ascontiguousarray(lay.seq_lens[b_idx])).cuda(), msl, 0.088, ws,
                           k_scale=1 / 64, v_scale=1 / 64)
        return G.storage_bytes(out).reshape(len(b_idx), -1)

    full = run(list(range(lay.B)), lay.max_seq_len)
    for b in range(lay.B):
        assert np.array_equal(run([b], lay.M * g.P)[0], full[b])


def test_fp8_decode_llama8b_full_size_sampled():
    """The full Llama-3-8B-shaped batch (B=231) over fp8 pools, launched as the
    benchmark launches it; the oracle recomputes a sample of sequences one by one."""
    torch = G.torch_mod()
    B, ks, vs = 231, 1 / 64, 1 / 64
    lay = W.llama8b_decode(B, seed=0)
    g = lay.geom
    kb, vb = W.device_pools(lay, seed=31)
    # codes from torch's own float -> e4m3 conversion after clamping (NaN slots stay NaN codes)
    kp = (kb.float() / ks).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    vp = (vb.float() / vs).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    del kb, vb
    q, k_new, v_new = W.device_step_values(lay, seed=32)
    order = np.argsort(lay.seq_lens)
    seqs = sorted(set(order[:3].tolist() + order[-3:].tolist() + order[:: B // 8].tolist()))
    P = g.P
    nb = [-(-int(lay.seq_lens[b]) // P) for b in seqs]
    used = np.unique(np.concatenate([lay.block_tables[b, :n] for b, n in zip(seqs, nb)]))
    remap = {int(x): i for i, x in enumerate(used)}
    idx = torch.from_numpy(used.astype(np.int64)).cuda()
    hk = kp.index_select(0, idx).cpu().numpy()          # oracle inputs, before this step's scatter
    hv = vp.index_select(0, idx).cpu().numpy()
    hbt = np.zeros((len(seqs), max(nb)), np.int32)
    for i, (b, n) in enumerate(zip(seqs, nb)):
        hbt[i, :n] = [remap[int(x)] for x in lay.block_tables[b, :n]]
    st = G.dev_status()
    wf.wf_reshape_and_cache(k_new, v_new, kp, vp, torch.from_numpy(lay.new_slots()).cuda(), st, k_scale=ks,
                            v_scale=vs)
    out = torch.empty_like(q)
    ws = torch.empty(wf.wf_paged_decode_workspace_size(B, g.H_q, lay.max_seq_len, wf.pool_desc(kp, ks, vs)),
                     dtype=torch.uint8, device="cuda")
    wf.wf_paged_decode(out, q, kp, vp, torch.from_numpy(lay.block_tables).cuda(),
                       torch.from_numpy(lay.seq_lens).cuda(), lay.max_seq_len, 1 / math.sqrt(g.D), ws, st,
                       k_scale=ks, v_scale=vs)
    assert wf.wf_device_status_fetch(st) == 0
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    sub = W.Layout(W.Geometry(g.H_q, g.H_kv, g.D, g.P, hk.shape[0], g.dtype), lay.seq_lens[seqs],
                   np.ones(len(seqs), np.int32), hbt, 0)
    oracle.reshape_and_cache_fp8(bits(k_new[seqs]), bits(v_new[seqs]), hk, hv, sub.new_slots(), ks, vs)
    ref = oracle.paged_decode_fp8(bits(q[seqs]), hk, hv, hbt, lay.seq_lens[seqs], 1 / math.sqrt(g.D), ks, vs)
    G.assert_close(G.from_dev(out[seqs], W.BF16), ref, W.BF16, "fp8 llama8b B=231")
    assert torch.isfinite(out.float()).all()


def test_fp8_decode_flags_bad_block():
    torch = G.torch_mod()
    lay = W.custom_layout(32, 8, 128, 16, W.BF16, [40, 50, 60], seed=30)
    vals = W.draw_layer_values(lay, np.random.default_rng(30))
    (dk, dv), (hk, hv) = _pools_both(lay, vals, 0.02, 0.02)
    bt = lay.block_tables.copy()
    bt[2, 1] = lay.geom.N + 7
    q = G.to_dev(vals.q, W.BF16)
    out = torch.empty_like(q)
    ws = torch.empty(wf.wf_paged_decode_workspace_size(lay.B, 32, lay.max_seq_len, wf.pool_desc(dk, 0.02, 0.02)),
                     dtype=torch.uint8, device="cuda")
    st = G.dev_status()
    wf.wf_paged_decode(out, q, dk, dv, torch.from_numpy(bt).cuda(), torch.from_numpy(lay.seq_lens).cuda(),
                       lay.max_seq_len, 0.088, ws, st, k_scale=0.02, v_scale=0.02)
    assert wf.wf_device_status_fetch(st) & wf.WF_DEV_BAD_BLOCK
    ref = oracle.paged_decode_fp8(vals.q, hk, hv, lay.block_tables, lay.seq_lens, 0.088, 0.02, 0.02)
    G.assert_close(G.from_dev(out[:2], W.BF16), ref[:2], W.BF16, "sequences with good tables")


def test_fp8_copy_blocks_is_a_byte_copy():
    torch = G.torch_mod()
    g = W.Geometry(H_q=8, H_kv=8, D=128, P=16, N=40, dtype=W.BF16)
    rng = np.random.default_rng(5)
    hk = rng.integers(0, 256, (g.N, g.P, g.H_kv, g.D), dtype=np.uint8)
    hv = rng.integers(0, 256, (g.N, g.P, g.H_kv, g.D), dtype=np.uint8)
    perm = rng.permutation(g.N).astype(np.int32)
    pairs = np.stack([perm[:9], perm[9:18]], axis=1)
    dk, dv = _dev_u8(hk), _dev_u8(hv)
    wf.wf_copy_blocks(dk, dv, torch.from_numpy(pairs).cuda(), k_scale=0.1, v_scale=0.1)
    oracle.copy_blocks(hk, hv, pairs, "fp8")
    assert np.array_equal(dk.cpu().numpy(), hk) and np.array_equal(dv.cpu().numpy(), hv)


def test_fp8_decode_flags_bad_seq_len():
    torch = G.torch_mod()
    lay = W.custom_layout(32, 8, 128, 16, W.BF16, [40, 300, 60, 17], seed=31)
    vals = W.draw_layer_values(lay, np.random.default_rng(31))
    (dk, dv), (hk, hv) = _pools_both(lay, vals, 0.02, 0.02)
    sl = lay.seq_lens.copy()
    sl[1] = 9999                                          # > max_seq_len: skipped and flagged
    q = G.to_dev(vals.q, W.BF16)
    out = torch.zeros_like(q)
    ws = torch.empty(wf.wf_paged_decode_workspace_size(lay.B, 32, lay.max_seq_len, wf.pool_desc(dk, 0.02, 0.02)),
                     dtype=torch.uint8, device="cuda")
    st = G.dev_status()
    wf.wf_paged_decode(out, q, dk, dv, torch.from_numpy(lay.block_tables).cuda(), torch.from_numpy(sl).cuda(),
                       lay.max_seq_len, 0.088, ws, st, k_scale=0.02, v_scale=0.02)
    assert wf.wf_device_status_fetch(st) == wf.WF_DEV_BAD_SEQLEN
    ref = oracle.paged_decode_fp8(vals.q, hk, hv, lay.block_tables, lay.seq_lens, 0.088, 0.02, 0.02)
    G.assert_close(G.from_dev(out[[0, 2, 3]], W.BF16), ref[[0, 2, 3]], W.BF16, "sequences with good lengths")


# one scale per KV head: spread over three octaves and not powers of two
def _head_scales(H_kv):
    return ([1 / 64 * (1.37 ** (h - 4)) for h in range(H_kv)], [1 / 96 * (0.71 ** (h - 3)) for h in range(H_kv)])


K_HEAD, V_HEAD = _head_scales(8)


def test_fp8_per_head_scatter_bit_exact():
    torch = G.torch_mod()
    T, N, P = 200, 20, 16
    rng = np.random.default_rng(17)
    x = rng.standard_normal((2, T, 8, 128)).astype(np.float32)
    x[:, ::9] *= 40.0                                   # saturate some codes in the small-scale heads
    k, v = W.f32_to_bf16_bits(x[0]), W.f32_to_bf16_bits(x[1])
    slots = rng.permutation(N * P)[:T].astype(np.int64)
    g = W.Geometry(H_q=8, H_kv=8, D=128, P=P, N=N, dtype=W.BF16)
    hk, hv = _empty_codes(g), _empty_codes(g)
    dk, dv = _dev_u8(hk), _dev_u8(hv)
    st = G.dev_status()
    wf.wf_reshape_and_cache(G.to_dev(k, W.BF16), G.to_dev(v, W.BF16), dk, dv, torch.from_numpy(slots).cuda(), st,
                            k_scale=K_HEAD, v_scale=V_HEAD)
    oracle.reshape_and_cache_fp8(k, v, hk, hv, slots, K_HEAD, V_HEAD)
    assert np.array_equal(dk.cpu().numpy(), hk) and np.array_equal(dv.cpu().numpy(), hv)
    assert wf.wf_device_status_fetch(st) == 0


@pytest.mark.parametrize("name", ["gqa4_ragged", "gqa2_P32", "core_mha12_D64", "gqa4_D64"])
def test_fp8_per_head_decode_matches_oracle(name):
    torch = G.torch_mod()
    lay = CASES[name]()
    vals = W.draw_layer_values(lay, np.random.default_rng(43))
    g = lay.geom
    scale = G.default_scale(g.D)
    st = G.dev_status()
    kh, vh = _head_scales(g.H_kv)
    (dk, dv), (hk, hv) = _pools_both(lay, vals, kh, vh, st)
    assert np.array_equal(dk.cpu().numpy(), hk) and np.array_equal(dv.cpu().numpy(), hv)
    q = G.to_dev(vals.q, W.BF16)
    out = torch.empty_like(q)
    ws = torch.empty(wf.wf_paged_decode_workspace_size(lay.B, g.H_q, lay.max_seq_len,
                                                       wf.pool_desc(dk, kh, vh)),
                     dtype=torch.uint8, device="cuda")
    wf.wf_paged_decode(out, q, dk, dv, torch.from_numpy(lay.block_tables).cuda(),
                       torch.from_numpy(lay.seq_lens).cuda(), lay.max_seq_len, scale, ws, st,
                       k_scale=kh, v_scale=vh)
    assert wf.wf_device_status_fetch(st) == 0
    ref = oracle.paged_decode_fp8(vals.q, hk, hv, lay.block_tables, lay.seq_lens, scale, kh, vh)
    G.assert_close(G.from_dev(out, W.BF16), ref, W.BF16, f"fp8 per-head {name}")

"""wf_copy_blocks on the GPU: whole pools bit-exact against the oracle's copy, and
prefix sharing with copy-on-write end to end (scatter, copy, scatter, decode)."""
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


def _pairs(N, n, rng):
    """n pairs with distinct destinations, none of which is a source."""
    perm = rng.permutation(N).astype(np.int32)
    return np.stack([perm[:n], perm[n:2 * n]], axis=1)


@pytest.mark.parametrize("H_kv,D,P,dtype,N,n", [
    (8, 128, 16, W.BF16, 300, 120),      # Llama-3-8B block (32 KB)
    (2, 64, 3, W.F32, 40, 13),           # odd block size, fp32
    (12, 64, 64, W.BF16, 9, 4),          # MHA, large block
    (4, 64, 1, W.BF16, 50, 1),           # one pair, one-slot blocks
])
def test_copy_blocks_whole_pool_bit_exact(H_kv, D, P, dtype, N, n):
    torch = G.torch_mod()
    g = W.Geometry(H_q=H_kv, H_kv=H_kv, D=D, P=P, N=N, dtype=dtype)
    rng = np.random.default_rng(N + n)
    kh = W._draw(rng, (N, P, H_kv, D), dtype, 1.0)
    vh = W._draw(rng, (N, P, H_kv, D), dtype, 1.0)
    pairs = _pairs(N, n, rng)
    kp, vp = G.to_dev(kh, dtype), G.to_dev(vh, dtype)
    st = G.dev_status()
    wf.wf_copy_blocks(kp, vp, torch.from_numpy(pairs).cuda(), st)
    oracle.copy_blocks(kh, vh, pairs, dtype)
    assert np.array_equal(G.storage_bytes(kp), kh.view(np.uint8).reshape(-1))
    assert np.array_equal(G.storage_bytes(vp), vh.view(np.uint8).reshape(-1))
    assert wf.wf_device_status_fetch(st) == 0


def test_copy_blocks_flags_bad_ids_and_copies_the_rest():
    torch = G.torch_mod()
    g = W.Geometry(H_q=2, H_kv=2, D=64, P=4, N=8, dtype=W.BF16)
    rng = np.random.default_rng(9)
    kh = W._draw(rng, (g.N, g.P, g.H_kv, g.D), g.dtype, 1.0)
    vh = W._draw(rng, (g.N, g.P, g.H_kv, g.D), g.dtype, 1.0)
    pairs = np.array([[0, 5], [1, 8], [-1, 6], [2, 7]], np.int32)   # the middle two are invalid
    kp, vp = G.to_dev(kh, g.dtype), G.to_dev(vh, g.dtype)
    st = G.dev_status()
    wf.wf_copy_blocks(kp, vp, torch.from_numpy(pairs).cuda(), st)
    oracle.copy_blocks(kh, vh, pairs[[0, 3]], g.dtype)
    assert np.array_equal(G.storage_bytes(kp), kh.view(np.uint8).reshape(-1))
    assert np.array_equal(G.storage_bytes(vp), vh.view(np.uint8).reshape(-1))
    assert wf.wf_device_status_fetch(st) & wf.WF_DEV_BAD_BLOCK


@pytest.mark.parametrize("prefix_len,H_q,H_kv,D,P", [
    (37, 32, 8, 128, 16),     # shared partial tail: tensor-core decode path
    (48, 32, 8, 128, 16),     # prefix ends on a block boundary: no copy needed
    (70, 8, 2, 64, 7),        # CUDA-core decode path, odd block size
])
def test_prefix_sharing_copy_on_write_end_to_end(prefix_len, H_q, H_kv, D, P):
    """Requests share prefix blocks; sharers copy the partial tail block, then every
    request writes its new token and decodes.  Pools bit-exact and outputs within
    the bf16 tolerance of the oracle doing the same steps."""
    torch = G.torch_mod()
    step = W.shared_prefix_step(H_q, H_kv, D, P, W.BF16, n_req=5, prefix_len=prefix_len, seed=prefix_len)
    vals = W.draw_shared_prefix_values(step, np.random.default_rng(11))
    g, post, c = step.geom, step.post, step.prefix_len
    scale = 1.0 / math.sqrt(D)
    st = G.dev_status()
    kp, vp = G.empty_dev_pool(g), G.empty_dev_pool(g)
    wf.wf_reshape_and_cache(G.to_dev(vals.k_prefix[:c], g.dtype), G.to_dev(vals.v_prefix[:c], g.dtype), kp, vp,
                            torch.from_numpy(step.prefix_slots).cuda(), st)
    if step.cow_pairs.shape[0]:
        wf.wf_copy_blocks(kp, vp, torch.from_numpy(step.cow_pairs).cuda(), st)
    wf.wf_reshape_and_cache(G.to_dev(vals.k_new, g.dtype), G.to_dev(vals.v_new, g.dtype), kp, vp,
                            torch.from_numpy(post.new_slots()).cuda(), st)
    out = G.run_decode(post, vals, (kp, vp), scale, st)
    # the oracle, same steps
    kh, vh = W.empty_pool(g), W.empty_pool(g)
    oracle.reshape_and_cache(vals.k_prefix[:c], vals.v_prefix[:c], kh, vh, step.prefix_slots, g.dtype)
    oracle.copy_blocks(kh, vh, step.cow_pairs, g.dtype)
    oracle.reshape_and_cache(vals.k_new, vals.v_new, kh, vh, post.new_slots(), g.dtype)
    assert np.array_equal(G.storage_bytes(kp), kh.view(np.uint8).reshape(-1))
    assert np.array_equal(G.storage_bytes(vp), vh.view(np.uint8).reshape(-1))
    ref = oracle.paged_decode(vals.q, kh, vh, post.block_tables, post.seq_lens, scale, g.dtype)
    G.assert_close(G.from_dev(out, W.BF16), ref, W.BF16, f"cow prefix {prefix_len}")
    assert wf.wf_device_status_fetch(st) == 0

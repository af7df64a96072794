"""wf_reshape_and_cache on the GPU against the oracle's scatter: whole pools bit-exact."""
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


def _layouts():
    return {
        "tiny": W.tiny_decode(0),
        "gpt2": W.gpt2_decode(0),
        "llama1b": W.llama1b_decode(0),
        "odd_P3_prefill": W.custom_layout(6, 3, 128, 3, W.BF16, [40, 7, 1], [5, 7, 1], seed=4),
        "P1_f32": W.custom_layout(4, 4, 64, 1, W.F32, [9, 3], seed=5),
        "P64_mha": W.custom_layout(12, 12, 64, 64, W.BF16, [100, 130, 64], seed=6),
        "P256_gqa4": W.custom_layout(32, 8, 128, 256, W.BF16, [600, 1, 257], seed=7),
        "P1024_largest_block": W.custom_layout(4, 2, 64, 1024, W.BF16, [1500, 3], seed=8),
    }


@pytest.mark.parametrize("name", list(_layouts().keys()))
def test_scatter_whole_pool_bit_exact(name):
    lay = _layouts()[name]
    vals = W.draw_layer_values(lay, np.random.default_rng(21))
    st = G.dev_status()
    kp, vp = G.build_dev_pools(lay, vals, st)
    kref, vref = oracle.build_pools(lay, vals)
    assert np.array_equal(G.storage_bytes(kp), kref.view(np.uint8).reshape(-1))
    assert np.array_equal(G.storage_bytes(vp), vref.view(np.uint8).reshape(-1))
    assert wf.wf_device_status_fetch(st) == 0


def test_scatter_mixed_step_bit_exact():
    """Mixed step: prefill and decode tokens written in one call through one pool."""
    pf, dc = W.mixed_step(0)
    torch = G.torch_mod()
    g = pf.geom
    rng = np.random.default_rng(3)
    slots = np.concatenate([pf.new_slots(), dc.new_slots()])
    T = slots.shape[0]
    k = W.f32_to_bf16_bits(rng.standard_normal((T, g.H_kv, g.D), dtype=np.float32))
    v = W.f32_to_bf16_bits(rng.standard_normal((T, g.H_kv, g.D), dtype=np.float32))
    kp = G.empty_dev_pool(g)
    vp = G.empty_dev_pool(g)
    st = G.dev_status()
    wf.wf_reshape_and_cache(G.to_dev(k, g.dtype), G.to_dev(v, g.dtype), kp, vp,
                            torch.from_numpy(slots).cuda(), st)
    kref = W.empty_pool(g)
    vref = W.empty_pool(g)
    oracle.reshape_and_cache(k, v, kref, vref, slots, g.dtype)
    assert np.array_equal(G.storage_bytes(kp), kref.view(np.uint8).reshape(-1))
    assert np.array_equal(G.storage_bytes(vp), vref.view(np.uint8).reshape(-1))
    assert wf.wf_device_status_fetch(st) == 0


def test_scatter_padding_and_out_of_range_slots():
    torch = G.torch_mod()
    g = W.Geometry(H_q=2, H_kv=2, D=64, P=4, N=6, dtype=W.BF16)
    rng = np.random.default_rng(0)
    k = W.f32_to_bf16_bits(rng.standard_normal((5, 2, 64), dtype=np.float32))
    v = W.f32_to_bf16_bits(rng.standard_normal((5, 2, 64), dtype=np.float32))
    slots = np.array([3, -1, 23, 24, 0], np.int64)     # 24 == N*P: out of range
    kp = G.empty_dev_pool(g)
    vp = G.empty_dev_pool(g)
    st = G.dev_status()
    wf.wf_reshape_and_cache(G.to_dev(k, g.dtype), G.to_dev(v, g.dtype), kp, vp,
                            torch.from_numpy(slots).cuda(), st)
    assert wf.wf_device_status_fetch(st) == wf.WF_DEV_BAD_SLOT
    keep = slots.copy()
    keep[3] = -1                                       # the oracle rejects it; compare the rest
    kref = W.empty_pool(g)
    vref = W.empty_pool(g)
    oracle.reshape_and_cache(k, v, kref, vref, keep, g.dtype)
    assert np.array_equal(G.storage_bytes(kp), kref.view(np.uint8).reshape(-1))
    assert np.array_equal(G.storage_bytes(vp), vref.view(np.uint8).reshape(-1))


def test_scatter_zero_tokens_is_a_no_op():
    torch = G.torch_mod()
    g = W.Geometry(H_q=2, H_kv=2, D=128, P=16, N=2, dtype=W.F32)
    kp = G.empty_dev_pool(g)
    vp = G.empty_dev_pool(g)
    e = torch.empty((0, 2, 128), dtype=torch.float32, device="cuda")
    wf.wf_reshape_and_cache(e, e, kp, vp, torch.empty(0, dtype=torch.int64, device="cuda"))
    assert torch.isnan(kp).all() and torch.isnan(vp).all()

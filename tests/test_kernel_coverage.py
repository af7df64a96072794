"""Every instance of the tensor-core kernels meets the oracle in some GPU case.

Host-only: asks libwf which kernel each GPU parity case reaches
(wf_paged_decode_kernel / wf_paged_prefill_kernel, no CUDA call) and checks that
the cases name every (group size G, head dim D) instance of the tensor-core
decode and prefill kernels, and the block sizes that change how a tile maps onto
a block (P = 16, 32 and 64 at D = 128).
"""
import pytest

from paged_kv_cache_wf_gb300 import binding as wf
from tests import _gpu as G


@pytest.fixture(scope="module")
def lib():
    return wf.load()


def _decode_cases():
    from tests import test_decode_gpu, test_fp8_gpu
    bf = {n: f().geom for n, f in test_decode_gpu.CASES.items()}
    f8 = {n: f().geom for n, f in test_fp8_gpu.CASES.items()}
    return bf, f8


def test_bf16_decode_cases_reach_every_tensor_core_instance(lib):
    bf, _ = _decode_cases()
    reached, heads_per_box = set(), set()
    for name, g in bf.items():
        if G.decode_kernel(g) == wf.WF_KERNEL_TENSOR_CORES:
            reached.add((g.H_q // g.H_kv, g.D))
            ht = 8
            while g.H_kv % ht:
                ht //= 2
            heads_per_box.add((ht, g.H_kv // ht > 1))
    assert {(gs, d) for gs in (1, 2, 4) for d in (64, 128)} <= reached, reached
    # every box shape (HT heads x 16 positions, 8 / HT boxes a tile), with one and
    # with several head groups per split
    assert {1, 2, 4, 8} <= {ht for ht, _ in heads_per_box}, heads_per_box
    assert {True, False} <= {many for _, many in heads_per_box}, heads_per_box
    p128 = {g.P for g in bf.values() if G.decode_kernel(g) == wf.WF_KERNEL_TENSOR_CORES and g.D == 128}
    assert {16, 32, 64} <= p128, p128
    # groups of 8 and fp32 pools run on the CUDA cores
    assert any(G.decode_kernel(g) == wf.WF_KERNEL_CUDA_CORES and g.H_q // g.H_kv == 8 and g.dtype == "bf16"
               for g in bf.values())


def test_fp8_decode_cases_reach_every_tensor_core_instance(lib):
    _, f8 = _decode_cases()
    reached = set()
    for g in f8.values():
        if G.decode_kernel(g, wf.WF_DTYPE_FP8_E4M3) == wf.WF_KERNEL_TENSOR_CORES:
            reached.add((g.H_q // g.H_kv, g.D))
    assert {(2, 64), (4, 64), (2, 128), (4, 128)} <= reached, reached
    assert any(G.decode_kernel(g, wf.WF_DTYPE_FP8_E4M3) == wf.WF_KERNEL_CUDA_CORES for g in f8.values())


def test_prefill_cases_reach_every_tensor_core_instance(lib):
    from paged_kv_cache_wf_gb300 import workloads as W
    from tests import test_prefill_gpu
    reached, simple = set(), 0
    for name, (H_q, H_kv, D, P, sl, ql) in test_prefill_gpu.CASES.items():
        g = W.custom_layout(H_q, H_kv, D, P, W.BF16, sl, ql, seed=len(name)).geom
        k = G.prefill_kernel(g)
        if k == wf.WF_KERNEL_TENSOR_CORES:
            reached.add((H_q // H_kv, D))
        elif k == wf.WF_KERNEL_TENSOR_CORES_SIMPLE:
            simple += 1
    want = {(gs, d) for gs in (1, 2, 4, 8) for d in (64, 128)}
    assert want <= reached, want - reached
    assert simple >= 2


def test_prefill_cases_reach_both_grids(lib):
    """The prefill cases run the persistent grid at every (G, D) instance, and the
    one-CTA-per-block grid (the list build's limits exceeded) at every instance too."""
    from paged_kv_cache_wf_gb300 import workloads as W
    from tests import test_prefill_gpu as T
    persistent, per_block = set(), set()
    for name, (H_q, H_kv, D, P, sl, ql) in T.CASES.items():
        lay = W.custom_layout(H_q, H_kv, D, P, W.BF16, sl, ql, seed=len(name))
        if G.prefill_kernel(lay.geom) != wf.WF_KERNEL_TENSOR_CORES:
            continue
        (persistent if G.prefill_persistent(lay) else per_block).add((H_q // H_kv, D))
    for D, grp in T.LEGACY_GRID:
        lay = T.legacy_grid_layout(D, grp)
        assert G.prefill_kernel(lay.geom) == wf.WF_KERNEL_TENSOR_CORES
        assert not G.prefill_persistent(lay)
        per_block.add((grp, D))
    want = {(gs, d) for gs in (1, 2, 4, 8) for d in (64, 128)}
    assert want <= persistent, want - persistent
    assert want <= per_block, want - per_block


def test_prefill_grid_query_limits(lib):
    """The list build takes up to 1024 requests and 4096 (request, query block) pairs;
    the query answers 0 for what the per-block grid or no tensor-core kernel runs."""
    d = wf.wf_pool_desc(64, 16, 8, 128, wf.WF_DTYPE_BF16, 1.0, 1.0)
    assert wf.wf_paged_prefill_persistent(d, 32, 1, 1)
    assert wf.wf_paged_prefill_persistent(d, 32, 1024, 1)
    assert not wf.wf_paged_prefill_persistent(d, 32, 1025, 1)
    assert not wf.wf_paged_prefill_persistent(d, 32, 0, 1)
    # G = 4: 256-row query blocks of 64 positions; 64 requests x 64 blocks = 4096 pairs
    assert wf.wf_paged_prefill_persistent(d, 32, 64, 64 * 64)
    assert not wf.wf_paged_prefill_persistent(d, 32, 64, 64 * 64 + 1)
    d.block_size = 8                                             # not a multiple of 16
    assert not wf.wf_paged_prefill_persistent(d, 32, 4, 100)
    d.block_size = 16
    d.dtype = wf.WF_DTYPE_FP8_E4M3                               # prefill is bf16 only
    assert not wf.wf_paged_prefill_persistent(d, 32, 4, 100)


def test_kernel_query_rejects_invalid_geometry(lib):
    d = wf.wf_pool_desc(16, 16, 8, 96, wf.WF_DTYPE_BF16, 1.0, 1.0)
    assert wf.wf_paged_decode_kernel(d, 32) == wf.WF_KERNEL_NONE
    d = wf.wf_pool_desc(16, 16, 8, 128, wf.WF_DTYPE_BF16, 1.0, 1.0)
    assert wf.wf_paged_decode_kernel(d, 12) == wf.WF_KERNEL_NONE   # 12 % 8 != 0
    assert wf.wf_paged_decode_kernel(d, 32) == wf.WF_KERNEL_TENSOR_CORES
    d.dtype = wf.WF_DTYPE_F32
    assert wf.wf_paged_decode_kernel(d, 32) == wf.WF_KERNEL_CUDA_CORES
    assert wf.wf_paged_prefill_kernel(d, 32) == wf.WF_KERNEL_NONE   # prefill is bf16 only

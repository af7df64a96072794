"""wf_paged_decode_static_scratch: paged decode for callers that cannot allocate.

Some callers cannot call cudaMalloc when they run attention (an allocator that
must not re-enter itself, a plugin whose host owns all device memory, a runtime
that fixes its memory at start-up).  This entry point uses the library's own
fixed device array as the decode workspace.  The tests call it through the C ABI
several times in a row, on different batches and pool formats, and check that:
  - its output bytes equal those of wf_paged_decode given a caller-allocated
    workspace (the same kernels run on the same geometry, so the bytes match
    exactly, which also catches a wrong offset inside the shared array);
  - a call after the first one leaves the device's free memory unchanged.
The file is named to be collected last.
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


def _static_call(lib, out, q, kp, vp, bt, sl, max_seq_len, scale, desc, status):
    torch = G.torch_mod()
    return lib.wf_paged_decode_static_scratch(
        out.data_ptr(), q.data_ptr(), kp.data_ptr(), vp.data_ptr(), bt.data_ptr(), int(bt.shape[1]),
        sl.data_ptr(), int(q.shape[0]), int(max_seq_len), int(q.shape[1]), float(scale), desc,
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _bf16_batch(lay, seed):
    vals = W.draw_layer_values(lay, np.random.default_rng(seed))
    kp, vp = G.build_dev_pools(lay, vals)
    return G.to_dev(vals.q, lay.geom.dtype), kp, vp, wf.pool_desc(kp), {}


def _fp8_batch(lay, seed, ks=1 / 64, vs=1 / 96):
    """Pools of e4m3 codes written by the library's quantising scatter."""
    torch = G.torch_mod()
    g = lay.geom
    vals = W.draw_layer_values(lay, np.random.default_rng(seed))
    kp = torch.full((g.N, g.P, g.H_kv, g.D), 0x7F, dtype=torch.uint8, device="cuda")
    vp = kp.clone()
    for k, v, s in ((vals.k_prefix, vals.v_prefix, lay.prefix_slots()), (vals.k_new, vals.v_new, lay.new_slots())):
        if k.shape[0]:
            wf.wf_reshape_and_cache(G.to_dev(k, W.BF16), G.to_dev(v, W.BF16), kp, vp, torch.from_numpy(s).cuda(),
                                    k_scale=ks, v_scale=vs)
    return G.to_dev(vals.q, W.BF16), kp, vp, wf.pool_desc(kp, ks, vs), dict(k_scale=ks, v_scale=vs)


def test_static_scratch_decode_equals_workspace_decode_on_calls_in_a_row():
    torch = G.torch_mod()
    lib = wf.load()
    batches = [
        ("llama1b bf16", W.llama1b_decode(0), _bf16_batch),
        ("llama8b heads bf16", W.custom_layout(32, 8, 128, 16, W.BF16, [1, 77, 1000, 129, 2500], seed=3),
         _bf16_batch),
        ("llama8b heads fp8", W.custom_layout(32, 8, 128, 16, W.BF16, [1, 300, 2049, 256, 257], seed=4), _fp8_batch),
        ("gpt2 bf16", W.gpt2_decode(0), _bf16_batch),
    ]
    for i, (name, lay, make) in enumerate(batches):
        q, kp, vp, desc, scales = make(lay, 100 + i)
        bt = torch.from_numpy(lay.block_tables).cuda()
        sl = torch.from_numpy(lay.seq_lens).cuda()
        scale = 1.0 / math.sqrt(lay.geom.D)
        need = wf.wf_paged_decode_workspace_size(lay.B, lay.geom.H_q, lay.max_seq_len, desc)
        assert 0 < need <= wf.WF_STATIC_SCRATCH_BYTES
        # reference: the existing entry point with a caller-allocated workspace
        ref = torch.empty_like(q)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        wf.wf_paged_decode(ref, q, kp, vp, bt, sl, lay.max_seq_len, scale, ws, **scales)
        # the static-scratch entry point, through the C ABI; everything it is given
        # exists before the free-memory reading
        out = torch.full_like(q, float("nan"))
        st = G.dev_status()
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = _static_call(lib, out, q, kp, vp, bt, sl, lay.max_seq_len, scale, desc, st)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert rc == wf.WF_OK, wf.status_string(rc)
        assert wf.wf_device_status_fetch(st) == 0
        assert np.array_equal(G.storage_bytes(out), G.storage_bytes(ref)), f"{name}: bytes differ"
        if i > 0:   # the first call may map the array (lazy module loading); later ones allocate nothing
            assert free_after == free_before, f"{name}: free memory {free_before} -> {free_after}"


def test_static_scratch_output_matches_oracle():
    """The static-scratch call on its own, against the fp64 oracle."""
    torch = G.torch_mod()
    lib = wf.load()
    lay = W.custom_layout(16, 8, 128, 16, W.BF16, [5, 600, 1300], seed=6)
    vals = W.draw_layer_values(lay, np.random.default_rng(6))
    kp, vp = G.build_dev_pools(lay, vals)
    q = G.to_dev(vals.q, W.BF16)
    out = torch.empty_like(q)
    st = G.dev_status()
    rc = _static_call(lib, out, q, kp, vp, torch.from_numpy(lay.block_tables).cuda(),
                      torch.from_numpy(lay.seq_lens).cuda(), lay.max_seq_len, 0.088, wf.pool_desc(kp), st)
    assert rc == wf.WF_OK
    assert wf.wf_device_status_fetch(st) == 0
    hk, hv = oracle.build_pools(lay, vals)
    ref = oracle.paged_decode(vals.q, hk, hv, lay.block_tables, lay.seq_lens, 0.088, W.BF16)
    G.assert_close(G.from_dev(out, W.BF16), ref, W.BF16, "static scratch vs oracle")


def test_static_scratch_rejects_batches_over_the_limit():
    torch = G.torch_mod()
    lib = wf.load()
    lay = W.llama8b_decode(231, seed=0)
    g = lay.geom
    d = wf.wf_pool_desc(g.N, g.P, g.H_kv, g.D, wf.WF_DTYPE_BF16)
    assert wf.wf_paged_decode_workspace_size(lay.B, g.H_q, lay.max_seq_len, d) > wf.WF_STATIC_SCRATCH_BYTES
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")  # never touched: rejected before launch
    p = small.data_ptr()
    rc = lib.wf_paged_decode_static_scratch(p, p, p, p, p, lay.M, p, lay.B, lay.max_seq_len, g.H_q, 0.088, d,
                                            None, torch.cuda.current_stream().cuda_stream)
    assert rc == wf.WF_ERR_WORKSPACE

"""wf_paged_decode_static_scratch: paged decode for callers that cannot allocate.

Some callers cannot call cudaMalloc when they run attention (an allocator that
must not re-enter itself, a plugin whose host owns all device memory, a runtime
that fixes its memory at start-up).  This entry point uses the library's own
fixed device array as the decode workspace.  The test calls it through the C ABI
twice in a row, on two different batches, and compares each result with
wf_paged_decode given a caller-allocated workspace, within the bf16 tolerance
the other decode tests use.  The file is named to be collected last.
"""
import math

import numpy as np
import pytest

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


def _batch(lay, seed):
    torch = G.torch_mod()
    vals = W.draw_layer_values(lay, np.random.default_rng(seed))
    kp, vp = G.build_dev_pools(lay, vals)
    q = G.to_dev(vals.q, lay.geom.dtype)
    bt = torch.from_numpy(lay.block_tables).cuda()
    sl = torch.from_numpy(lay.seq_lens).cuda()
    return q, kp, vp, bt, sl


def _static_call(lib, out, q, kp, vp, bt, sl, max_seq_len, scale, status):
    torch = G.torch_mod()
    return lib.wf_paged_decode_static_scratch(
        out.data_ptr(), q.data_ptr(), kp.data_ptr(), vp.data_ptr(), bt.data_ptr(), int(bt.shape[1]),
        sl.data_ptr(), int(q.shape[0]), int(max_seq_len), int(q.shape[1]), float(scale), wf.pool_desc(kp),
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_static_scratch_decode_matches_workspace_decode_twice():
    torch = G.torch_mod()
    lib = wf.load()
    batches = [W.llama1b_decode(0),
               W.custom_layout(32, 8, 128, 16, W.BF16, [1, 77, 1000, 129, 2500], seed=3)]
    for i, lay in enumerate(batches):
        q, kp, vp, bt, sl = _batch(lay, 100 + i)
        scale = 1.0 / math.sqrt(lay.geom.D)
        need = wf.wf_paged_decode_workspace_size(lay.B, lay.geom.H_q, lay.max_seq_len, wf.pool_desc(kp))
        assert 0 < need <= wf.WF_STATIC_SCRATCH_BYTES
        # reference: the existing entry point with a caller-allocated workspace
        ref = torch.empty_like(q)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        wf.wf_paged_decode(ref, q, kp, vp, bt, sl, lay.max_seq_len, scale, ws)
        # the static-scratch entry point, through the C ABI
        out = torch.full_like(q, float("nan"))
        st = G.dev_status()
        rc = _static_call(lib, out, q, kp, vp, bt, sl, lay.max_seq_len, scale, st)
        assert rc == wf.WF_OK, wf.status_string(rc)
        assert wf.wf_device_status_fetch(st) == 0
        G.assert_close(G.from_dev(out, lay.geom.dtype), G.from_dev(ref, lay.geom.dtype), lay.geom.dtype,
                       f"static-scratch call {i + 1}")


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

"""GPU-side helpers for the parity tests: move generated inputs to the device and
run the library's calls through the C ABI binding."""
import math

import numpy as np

from paged_kv_cache_wf_gb300 import binding as wf
from paged_kv_cache_wf_gb300 import workloads as W

TOL = {
    # spec tolerances against the fp64 oracle
    W.F32: dict(max_abs=1e-4, mean_abs=None),
    W.BF16: dict(max_abs=2e-2, mean_abs=2e-3),
}


def geom_desc(geom) -> "wf.wf_pool_desc":
    """The C pool descriptor of a workload geometry (no device memory needed)."""
    code = {W.F32: wf.WF_DTYPE_F32, W.BF16: wf.WF_DTYPE_BF16}.get(geom.dtype, wf.WF_DTYPE_FP8_E4M3)
    return wf.wf_pool_desc(geom.N, geom.P, geom.H_kv, geom.D, code, 1.0, 1.0)


def decode_kernel(geom, dtype_code=None) -> int:
    """WF_KERNEL_* of the kernel wf_paged_decode runs for this geometry."""
    d = geom_desc(geom)
    if dtype_code is not None:
        d.dtype = dtype_code
    return wf.wf_paged_decode_kernel(d, geom.H_q)


def prefill_kernel(geom) -> int:
    """WF_KERNEL_* of the kernel wf_paged_prefill runs for this geometry."""
    return wf.wf_paged_prefill_kernel(geom_desc(geom), geom.H_q)


def prefill_persistent(lay) -> bool:
    """Whether wf_paged_prefill runs this batch as the persistent grid."""
    return wf.wf_paged_prefill_persistent(geom_desc(lay.geom), lay.geom.H_q, lay.B, lay.max_q_len)


def torch_mod():
    import torch
    return torch


def to_dev(a: np.ndarray, dtype: str):
    torch = torch_mod()
    if dtype == W.F32:
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def from_dev(t, dtype: str) -> np.ndarray:
    """Device tensor in storage dtype -> float64 numpy (exact widening)."""
    torch = torch_mod()
    if dtype == W.F32:
        return t.detach().cpu().numpy().astype(np.float64)
    bits = t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def storage_bytes(t) -> np.ndarray:
    torch = torch_mod()
    return t.detach().contiguous().view(torch.uint8).cpu().numpy().reshape(-1)


def empty_dev_pool(geom):
    return to_dev(W.empty_pool(geom), geom.dtype)


def dev_status():
    torch = torch_mod()
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def build_dev_pools(layout, vals, status=None):
    """Device pools: NaN everywhere, then wf_reshape_and_cache of every prefix row
    and of this step's new rows (the GPU path's own scatter)."""
    torch = torch_mod()
    g = layout.geom
    kp = empty_dev_pool(g)
    vp = empty_dev_pool(g)
    if vals.k_prefix.shape[0]:
        wf.wf_reshape_and_cache(to_dev(vals.k_prefix, g.dtype), to_dev(vals.v_prefix, g.dtype), kp, vp,
                                torch.from_numpy(layout.prefix_slots()).cuda(), status)
    if vals.k_new.shape[0]:
        wf.wf_reshape_and_cache(to_dev(vals.k_new, g.dtype), to_dev(vals.v_new, g.dtype), kp, vp,
                                torch.from_numpy(layout.new_slots()).cuda(), status)
    return kp, vp


def run_decode(layout, vals, pools, scale, status=None, max_seq_len=None):
    torch = torch_mod()
    g = layout.geom
    kp, vp = pools
    q = to_dev(vals.q, g.dtype)
    out = torch.empty_like(q)
    msl = int(max_seq_len or layout.max_seq_len)
    ws_bytes = wf.wf_paged_decode_workspace_size(layout.B, g.H_q, msl, wf.pool_desc(kp))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    bt = torch.from_numpy(layout.block_tables).cuda()
    sl = torch.from_numpy(layout.seq_lens).cuda()
    wf.wf_paged_decode(out, q, kp, vp, bt, sl, msl, scale, ws, status)
    return out


def run_prefill(layout, vals, pools, scale, status=None):
    torch = torch_mod()
    g = layout.geom
    kp, vp = pools
    q = to_dev(vals.q, g.dtype)
    out = torch.empty_like(q)
    bt = torch.from_numpy(layout.block_tables).cuda()
    sl = torch.from_numpy(layout.seq_lens).cuda()
    cu = torch.from_numpy(layout.cu_q_lens).cuda()
    wf.wf_paged_prefill(out, q, kp, vp, bt, sl, cu, layout.max_q_len, layout.max_seq_len, scale, status)
    return out


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite outputs"
    err = np.abs(got - ref)
    tol = TOL[dtype]
    assert err.max() <= tol["max_abs"], f"{what}: max abs err {err.max():.3e} > {tol['max_abs']}"
    if tol["mean_abs"] is not None:
        assert err.mean() <= tol["mean_abs"], f"{what}: mean abs err {err.mean():.3e} > {tol['mean_abs']}"
    return float(err.max()), float(err.mean())


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)

"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports every
entry point include/wf.h declares, and rejects bad arguments before launching
anything (these calls return before any CUDA call, so no GPU is needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_cache_wf_gb300 import binding as wf
from paged_kv_cache_wf_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # 16-byte aligned non-null address; never dereferenced by these calls


@pytest.fixture(scope="module")
def lib():
    build.build()
    return wf.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(wf_[a-z0-9_]+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.check_output(["nm", "-D", "--defined-only", build.LIB], text=True)
    exported = set(re.findall(r"\bT (wf_[a-z0-9_]+)", out))
    declared = _declared()
    assert declared, "no declarations found"
    assert declared <= exported, declared - exported
    assert declared == set(wf.EXPORTS)


def test_abi_version_and_status_strings(lib):
    assert lib.wf_abi_version() == 104
    for code in range(6):
        assert wf.status_string(code)


def _desc(N=10, P=16, H=2, D=64, dt=wf.WF_DTYPE_BF16, ks=0.0, vs=0.0):
    return wf.wf_pool_desc(N, P, H, D, dt, ks, vs)


def _fp8(N=10, P=16, H=8, D=128, ks=0.05, vs=0.05):
    return _desc(N, P, H, D, wf.WF_DTYPE_FP8_E4M3, ks, vs)


def test_scatter_argument_checks(lib):
    d = _desc()
    f = lib.wf_reshape_and_cache
    assert f(None, None, None, None, None, 0, d, None, None) == wf.WF_OK  # T = 0: no-op
    assert f(None, None, None, None, None, 3, d, None, None) == wf.WF_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, -1, d, None, None) == wf.WF_ERR_INVALID_ARG
    assert f(FAKE + 4, FAKE, FAKE, FAKE, FAKE, 3, d, None, None) == wf.WF_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 3, _desc(D=96), None, None) == wf.WF_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 3, _desc(dt=7), None, None) == wf.WF_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 3, _desc(P=0), None, None) == wf.WF_ERR_INVALID_ARG


def test_copy_blocks_argument_checks(lib):
    d = _desc()
    f = lib.wf_copy_blocks
    assert f(None, None, None, 0, d, None, None) == wf.WF_OK  # no pairs: no-op
    assert f(None, None, None, 2, d, None, None) == wf.WF_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, -1, d, None, None) == wf.WF_ERR_INVALID_ARG
    assert f(FAKE + 8, FAKE, FAKE, 2, d, None, None) == wf.WF_ERR_INVALID_ARG      # pool not 16-byte aligned
    assert f(FAKE, FAKE, FAKE + 2, 2, d, None, None) == wf.WF_ERR_INVALID_ARG      # pairs not 4-byte aligned
    assert f(FAKE, FAKE, FAKE, 2, _desc(D=96), None, None) == wf.WF_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, 2, _desc(N=0), None, None) == wf.WF_ERR_INVALID_ARG


def test_decode_workspace_size(lib):
    d = _desc(N=100, P=16, H=8, D=128)
    a = wf.wf_paged_decode_workspace_size(231, 32, 8704, d)
    b = wf.wf_paged_decode_workspace_size(231, 32, 128, d)
    assert a > b > 0
    assert wf.wf_paged_decode_workspace_size(4, 31, 100, d) == 0      # H_q % H_kv != 0
    assert wf.wf_paged_decode_workspace_size(4, 32, 0, d) == 0


def test_decode_argument_checks(lib):
    d = _desc(N=10, P=16, H=2, D=64)
    f = lib.wf_paged_decode
    ws = wf.wf_paged_decode_workspace_size(4, 8, 64, d)
    ok = dict(out=FAKE, q=FAKE, kp=FAKE, vp=FAKE, bt=FAKE, M=4, sl=FAKE, B=4, msl=64, Hq=8, scale=0.1,
              d=d, ws=FAKE, wsb=ws)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["out"], a["q"], a["kp"], a["vp"], a["bt"], a["M"], a["sl"], a["B"], a["msl"], a["Hq"],
                 a["scale"], a["d"], a["ws"], a["wsb"], None, None)

    assert call(B=0) == wf.WF_OK
    assert call(Hq=7) == wf.WF_ERR_INVALID_ARG                 # H_q % H_kv != 0
    assert call(Hq=18, d=_desc(N=10, P=16, H=2, D=64)) == wf.WF_ERR_UNSUPPORTED  # G = 9 > 8
    assert call(msl=65) == wf.WF_ERR_INVALID_ARG               # max_seq_len > M * P
    assert call(scale=float("inf")) == wf.WF_ERR_INVALID_ARG
    assert call(q=None) == wf.WF_ERR_INVALID_ARG
    assert call(out=FAKE + 8) == wf.WF_ERR_INVALID_ARG         # misaligned
    assert call(wsb=ws - 1) == wf.WF_ERR_WORKSPACE
    assert call(ws=None) == wf.WF_ERR_WORKSPACE
    assert call(d=_desc(D=80)) == wf.WF_ERR_UNSUPPORTED


def test_prefill_argument_checks(lib):
    d = _desc(N=10, P=16, H=2, D=128)
    f = lib.wf_paged_prefill

    def call(d=d, B=2, T=10, mq=8, msl=40, Hq=8, q=FAKE, cu=FAKE):
        return f(FAKE, q, FAKE, FAKE, FAKE, 4, FAKE, cu, B, T, mq, msl, Hq, 0.1, d, None, None)

    assert call(B=0) == wf.WF_OK
    assert call(T=0) == wf.WF_OK
    assert call(d=_desc(dt=wf.WF_DTYPE_F32, D=128)) == wf.WF_ERR_UNSUPPORTED   # bf16 only
    assert call(Hq=9) == wf.WF_ERR_INVALID_ARG
    assert call(msl=65) == wf.WF_ERR_INVALID_ARG
    assert call(mq=50) == wf.WF_ERR_INVALID_ARG                # max_q_len > max_seq_len
    assert call(cu=None) == wf.WF_ERR_INVALID_ARG
    assert call(q=FAKE + 2) == wf.WF_ERR_INVALID_ARG


def test_status_fetch_rejects_null(lib):
    assert lib.wf_device_status_fetch(None, None, 1, None) == wf.WF_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        wf.load.__wrapped__(str(tmp_path / "nope.so")) if hasattr(wf.load, "__wrapped__") else \
            _load_fresh(str(tmp_path / "nope.so"))


def _load_fresh(path):
    saved = wf._lib
    wf._lib = None
    try:
        return wf.load(path)
    finally:
        wf._lib = saved


def test_fp8_pool_argument_checks(lib):
    """fp8 e4m3 pools need finite positive scales; decode takes them in every
    geometry the bf16 path takes (tensor cores or CUDA cores); prefill does not
    take them."""
    sc = lib.wf_reshape_and_cache
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))):
        assert sc(FAKE, FAKE, FAKE, FAKE, FAKE, 0, _fp8(ks=ks, vs=vs), None, None) == wf.WF_ERR_INVALID_ARG
    assert sc(None, None, None, None, None, 0, _fp8(), None, None) == wf.WF_OK
    assert lib.wf_copy_blocks(FAKE, FAKE, FAKE, 0, _fp8(), None, None) == wf.WF_OK
    assert lib.wf_copy_blocks(FAKE, FAKE, FAKE, 0, _fp8(ks=0.0), None, None) == wf.WF_ERR_INVALID_ARG

    f = lib.wf_paged_decode

    def dec(d, Hq=32, B=0):
        ws = wf.wf_paged_decode_workspace_size(4, Hq, 64, d)
        return f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, B, 64, Hq, 0.1, d, FAKE, ws, None, None)

    assert dec(_fp8()) == wf.WF_OK                                    # G = 4: supported (B = 0: no-op)
    assert dec(_fp8(), Hq=16) == wf.WF_OK                             # G = 2
    assert dec(_fp8(), Hq=8) == wf.WF_OK                              # G = 1 (CUDA cores)
    assert dec(_fp8(), Hq=64) == wf.WF_OK                             # G = 8
    assert dec(_fp8(D=64)) == wf.WF_OK
    assert dec(_fp8(H=4), Hq=16) == wf.WF_OK
    assert dec(_fp8(P=24)) == wf.WF_OK                              # P % 16 != 0
    assert dec(_fp8(), Hq=72) == wf.WF_ERR_UNSUPPORTED                # G = 9, as for bf16
    assert dec(_fp8(D=96)) == wf.WF_ERR_UNSUPPORTED                   # as for bf16
    assert dec(_fp8(ks=0.0)) == wf.WF_ERR_INVALID_ARG

    pf = lib.wf_paged_prefill
    rc = pf(FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, 8, 8, 64, 32, 0.1, _fp8(), None, None)
    assert rc == wf.WF_ERR_UNSUPPORTED


def test_fp8_per_head_scale_checks(lib):
    """Per-head fp8 scales (host arrays of H_kv values) replace the per-tensor ones;
    each must be finite and positive, and at most 64 heads may carry them."""
    sc = lib.wf_reshape_and_cache

    def desc(ks, vs, H=8, k_scale=0.0, v_scale=0.0):
        d = _fp8(H=H, ks=k_scale, vs=v_scale)
        karr = (ctypes.c_float * len(ks))(*ks) if ks is not None else None
        varr = (ctypes.c_float * len(vs))(*vs) if vs is not None else None
        d.k_head_scales = ctypes.cast(karr, ctypes.POINTER(ctypes.c_float)) if karr is not None else None
        d.v_head_scales = ctypes.cast(varr, ctypes.POINTER(ctypes.c_float)) if varr is not None else None
        d._keep = (karr, varr)
        return d

    good = [0.01 * (h + 1) for h in range(8)]
    assert sc(None, None, None, None, None, 0, desc(good, good), None, None) == wf.WF_OK      # per-tensor unused
    assert sc(None, None, None, None, None, 0, desc(good, None), None, None) == wf.WF_ERR_INVALID_ARG  # v_scale 0
    assert sc(None, None, None, None, None, 0, desc(good, None, v_scale=0.5), None, None) == wf.WF_OK
    bad = list(good)
    bad[5] = 0.0
    assert sc(None, None, None, None, None, 0, desc(bad, good), None, None) == wf.WF_ERR_INVALID_ARG
    bad[5] = float("nan")
    assert sc(None, None, None, None, None, 0, desc(good, bad), None, None) == wf.WF_ERR_INVALID_ARG
    wide = [0.5] * 80
    assert sc(None, None, None, None, None, 0, desc(wide, wide, H=80), None, None) == wf.WF_ERR_UNSUPPORTED
    assert sc(None, None, None, None, None, 0, _fp8(H=80), None, None) == wf.WF_OK           # per-tensor: any H
    # the binding builds the arrays from a sequence
    import torch
    d = wf.pool_desc(torch.empty((2, 16, 8, 128), dtype=torch.uint8), good, 0.25)
    assert d.dtype == wf.WF_DTYPE_FP8_E4M3 and abs(d.k_head_scales[7] - 0.08) < 1e-7 and not d.v_head_scales


def test_static_scratch_checks_arguments_before_its_size_limit(lib):
    """wf_paged_decode_static_scratch applies wf_paged_decode's argument rules
    first; only a valid batch over WF_STATIC_SCRATCH_BYTES gets WF_ERR_WORKSPACE.
    None of these calls launches anything."""
    f = lib.wf_paged_decode_static_scratch
    d = _desc(N=4000, P=16, H=8, D=128)
    B, M, msl = 4096, 512, 8192          # far over the 32 MiB array
    assert wf.wf_paged_decode_workspace_size(B, 32, msl, d) > wf.WF_STATIC_SCRATCH_BYTES
    args = lambda scale, msl=msl, m=M, ptr=FAKE: (ptr, ptr, ptr, ptr, ptr, m, ptr, B, msl, 32, scale, d, None, None)
    assert f(*args(0.088)) == wf.WF_ERR_WORKSPACE
    assert f(*args(float("nan"))) == wf.WF_ERR_INVALID_ARG                 # non-finite scale
    assert f(*args(0.088, msl=M * 16 + 1)) == wf.WF_ERR_INVALID_ARG        # max_seq_len > M * P
    assert f(*args(0.088, m=0)) == wf.WF_ERR_INVALID_ARG                   # no table columns
    assert f(*args(0.088, ptr=FAKE + 4)) == wf.WF_ERR_INVALID_ARG          # misaligned pointers
    assert f(*args(0.088, ptr=None)) == wf.WF_ERR_INVALID_ARG              # null pointers
    empty = (None, None, None, None, None, 1, None, 0, 16, 32, 0.088, d, None, None)
    assert f(*empty) == wf.WF_OK                                            # empty batch: no-op


def test_decode_worker_argument_checks(lib):
    f = lib.wf_decode_worker
    d = _desc(N=10, P=16, H=2, D=64)
    ok = lambda **kw: dict(dict(out=FAKE, q=FAKE, rows=4, kp=FAKE, vp=FAKE, bt=FAKE, trows=4, M=2, hq=4, scale=0.1,
                                pool=d, tasks=FAKE, cap=8, mb=FAKE, workers=2, timeout=10**6), **kw)
    call = lambda a: f(a["out"], a["q"], a["rows"], a["kp"], a["vp"], a["bt"], a["trows"], a["M"], a["hq"],
                       a["scale"], a["pool"], a["tasks"], a["cap"], a["mb"], a["workers"], a["timeout"], None, None)
    assert call(ok(mb=None)) == wf.WF_ERR_INVALID_ARG
    assert call(ok(mb=FAKE + 4)) == wf.WF_ERR_INVALID_ARG            # mailbox not 16-byte aligned
    assert call(ok(workers=0)) == wf.WF_ERR_INVALID_ARG
    assert call(ok(timeout=0)) == wf.WF_ERR_INVALID_ARG
    assert call(ok(hq=3)) == wf.WF_ERR_INVALID_ARG                   # 3 % 2 != 0
    assert call(ok(hq=18)) == wf.WF_ERR_UNSUPPORTED                  # group of 9
    assert call(ok(scale=float("inf"))) == wf.WF_ERR_INVALID_ARG
    assert call(ok(pool=_fp8(N=10, P=16, H=2, D=64))) == wf.WF_ERR_UNSUPPORTED
    assert call(ok(tasks=None)) == wf.WF_ERR_INVALID_ARG


def test_prefill_decode_query_and_argument_checks(lib):
    d = _desc(N=100, P=16, H=8, D=128)
    assert lib.wf_paged_prefill_decode_fused(d, 32) == 1          # Llama-3-8B heads: one grid
    assert lib.wf_paged_prefill_decode_fused(d, 64) == 0          # a group of 8: two launches
    assert lib.wf_paged_prefill_decode_fused(_desc(N=100, P=16, H=2, D=128), 8) == 0   # H_kv not a multiple of 8
    assert lib.wf_paged_prefill_decode_fused(_desc(N=100, P=7, H=8, D=128), 32) == 0   # P % 16 != 0
    f = lib.wf_paged_prefill_decode
    F = FAKE
    ok = (F, F, F, 4, F, F, 2, 10, 8, 64, F, F, F, 4, F, 3, 64, F, F, 32, 0.088, d, None, 0, None, None)
    assert f(*ok) == wf.WF_ERR_WORKSPACE                          # a decode batch needs its workspace
    bad = list(ok); bad[20] = float("nan")
    assert f(*bad) == wf.WF_ERR_INVALID_ARG
    bad = list(ok); bad[9] = 4                                    # prefill max_seq_len < max_q_len
    assert f(*bad) == wf.WF_ERR_INVALID_ARG
    none = (None, None, None, 1, None, None, 0, 0, 0, 16, None, None, None, 1, None, 0, 16, None, None, 32, 0.088, d,
            None, 0, None, None)
    assert f(*none) == wf.WF_OK                                   # nothing to do

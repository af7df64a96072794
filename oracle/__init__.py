"""fp64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
(``__graft_entry__.smoke``) and the CPU-baseline leg of ``bench.py`` may import
this package.  It shares no code with the CUDA library: the arithmetic lives
in ``wfo.c`` (plain C, fp64), this file only builds it and marshals numpy
arrays.

Functions follow (page titles and sections):
  - weft, "Cache layouts" and "Shapes and symbols" (pool [N, P, H_kv, D],
    scatter through slot_mapping, gather through block_table, GQA);
  - ember, "The core idea, in one picture" (block_table[p // P], offset p % P);
  - tiny-vllm-py, "KV Cache" (decode attends to all cached positions including
    the new one; prefill is causal).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wfo.c")
_LIB_PATH = os.path.join(_HERE, "libwfo.so")
_lock = threading.Lock()
_lib = None

F32, BF16, FP8 = 0, 1, 2
_DTYPES = {"f32": F32, "bf16": BF16, "fp8": FP8}   # fp8: e4m3 codes, uint8 pools


def build(force: bool = False) -> str:
    """Compile wfo.c into libwfo.so with gcc (fp contraction off, no -march)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(os.path.join(_HERE, "wfo.h")))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            p, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.wfo_reshape_and_cache.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i32]
            lib.wfo_reshape_and_cache.restype = i32
            lib.wfo_copy_blocks.argtypes = [p, p, p, i64, i64, i64, i64, i64, i32]
            lib.wfo_copy_blocks.restype = i32
            f = ctypes.c_float
            lib.wfo_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.wfo_e4m3_decode.restype = d
            lib.wfo_e4m3_encode.argtypes = [f]
            lib.wfo_e4m3_encode.restype = ctypes.c_uint8
            lib.wfo_reshape_and_cache_fp8.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, p, p]
            lib.wfo_reshape_and_cache_fp8.restype = i32
            lib.wfo_paged_decode_fp8.argtypes = [p, p, p, p, p, i64, p, i64, i64, i64, i64, i64, i64,
                                                 d, p, p, i32]
            lib.wfo_paged_decode_fp8.restype = i32
            lib.wfo_paged_decode.argtypes = [p, p, p, p, p, i64, p, i64, i64, i64, i64, i64, i64,
                                             d, i32, i32]
            lib.wfo_paged_decode.restype = i32
            lib.wfo_paged_prefill.argtypes = [p, p, p, p, p, i64, p, p, i64, i64, i64, i64, i64,
                                              i64, d, i32, i32]
            lib.wfo_paged_prefill.restype = i32
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype=None):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} failed with code {rc}")


def default_threads() -> int:
    return os.cpu_count() or 1


def reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, dtype: str):
    """In-place scatter into (contiguous) numpy pools k_pool/v_pool [N, P, H_kv, D]."""
    lib = _load()
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    N, P, H_kv, D = k_pool.shape
    k = _c(k, k_pool.dtype)
    v = _c(v, v_pool.dtype)
    slots = _c(slot_mapping, np.int64)
    T = int(slots.shape[0])
    _check(lib.wfo_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool), _ptr(slots),
                                     T, N, P, H_kv, D, _DTYPES[dtype]), "wfo_reshape_and_cache")


def copy_blocks(k_pool, v_pool, pairs, dtype: str):
    """In-place copy-on-write block copy on numpy pools: block dst of both pools
    becomes block src as it was before the call, for every (src, dst) row of pairs."""
    lib = _load()
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    N, P, H_kv, D = k_pool.shape
    pr = _c(np.asarray(pairs).reshape(-1, 2), np.int32)
    _check(lib.wfo_copy_blocks(_ptr(k_pool), _ptr(v_pool), _ptr(pr), int(pr.shape[0]), N, P, H_kv, D,
                               _DTYPES[dtype]), "wfo_copy_blocks")


def e4m3_decode(code: int) -> float:
    return float(_load().wfo_e4m3_decode(int(code)))


def e4m3_encode(y: float) -> int:
    return int(_load().wfo_e4m3_encode(float(y)))


def head_scales(scale, H_kv: int) -> np.ndarray:
    """A per-tensor scale (a number) or H_kv per-head scales -> float32 [H_kv]."""
    a = np.asarray(scale, dtype=np.float32).reshape(-1)
    if a.shape[0] == 1:
        a = np.full(H_kv, a[0], np.float32)
    assert a.shape[0] == H_kv, (a.shape, H_kv)
    return np.ascontiguousarray(a)


def reshape_and_cache_fp8(k, v, k_pool, v_pool, slot_mapping, k_scale, v_scale):
    """In-place scatter of bf16 rows into uint8 (e4m3 code) pools [N, P, H_kv, D];
    k_scale, v_scale: one number or one scale per KV head."""
    lib = _load()
    assert k_pool.dtype == np.uint8 and k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    N, P, H_kv, D = k_pool.shape
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    slots = _c(slot_mapping, np.int64)
    ks, vs = head_scales(k_scale, H_kv), head_scales(v_scale, H_kv)
    _check(lib.wfo_reshape_and_cache_fp8(_ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool), _ptr(slots),
                                         int(slots.shape[0]), N, P, H_kv, D, _ptr(ks), _ptr(vs)),
           "wfo_reshape_and_cache_fp8")


def paged_decode_fp8(q, k_pool, v_pool, block_tables, seq_lens, scale: float, k_scale, v_scale,
                     nthreads: int | None = None) -> np.ndarray:
    """fp64 decode outputs [B, H_q, D] for bf16 q and e4m3-code pools (k_scale, v_scale:
    one number or one scale per KV head)."""
    lib = _load()
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, np.uint8)
    v_pool = _c(v_pool, np.uint8)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    B, H_q, D = q.shape
    N, P, H_kv, _ = k_pool.shape
    ks, vs = head_scales(k_scale, H_kv), head_scales(v_scale, H_kv)
    out = np.zeros((B, H_q, D), np.float64)
    _check(lib.wfo_paged_decode_fp8(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(bt), int(bt.shape[1]),
                                    _ptr(sl), B, H_q, H_kv, D, N, P, float(scale), _ptr(ks), _ptr(vs),
                                    nthreads or default_threads()), "wfo_paged_decode_fp8")
    return out


def paged_decode(q, k_pool, v_pool, block_tables, seq_lens, scale: float, dtype: str,
                 nthreads: int | None = None) -> np.ndarray:
    """fp64 decode outputs [B, H_q, D] for storage-dtype q [B, H_q, D] and pools."""
    lib = _load()
    q = _c(q)
    k_pool = _c(k_pool)
    v_pool = _c(v_pool)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    B, H_q, D = q.shape
    N, P, H_kv, D2 = k_pool.shape
    assert D == D2 and bt.shape[0] == B
    out = np.zeros((B, H_q, D), dtype=np.float64)
    _check(lib.wfo_paged_decode(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(bt),
                                bt.shape[1], _ptr(sl), B, H_q, H_kv, D, N, P, float(scale),
                                _DTYPES[dtype], nthreads or default_threads()),
           "wfo_paged_decode")
    return out


def paged_prefill(q, k_pool, v_pool, block_tables, seq_lens, cu_q_lens, scale: float,
                  dtype: str, nthreads: int | None = None) -> np.ndarray:
    """fp64 causal prefill outputs [T_total, H_q, D]."""
    lib = _load()
    q = _c(q)
    k_pool = _c(k_pool)
    v_pool = _c(v_pool)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    cu = _c(cu_q_lens, np.int32)
    T, H_q, D = q.shape
    N, P, H_kv, _ = k_pool.shape
    B = int(sl.shape[0])
    assert cu.shape[0] == B + 1 and int(cu[-1]) == T
    out = np.zeros((T, H_q, D), dtype=np.float64)
    _check(lib.wfo_paged_prefill(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(bt),
                                 bt.shape[1], _ptr(sl), _ptr(cu), B, H_q, H_kv, D, N, P,
                                 float(scale), _DTYPES[dtype], nthreads or default_threads()),
           "wfo_paged_prefill")
    return out


def build_pools(layout, vals):
    """Oracle-side pools for one layer: NaN everywhere, then the oracle's own
    scatter of every cached prefix row and every new row (the step's write)."""
    from paged_kv_cache_wf_gb300 import workloads as W  # generator only
    g = layout.geom
    k_pool = W.empty_pool(g)
    v_pool = W.empty_pool(g)
    reshape_and_cache(vals.k_prefix, vals.v_prefix, k_pool, v_pool, layout.prefix_slots(), g.dtype)
    reshape_and_cache(vals.k_new, vals.v_new, k_pool, v_pool, layout.new_slots(), g.dtype)
    return k_pool, v_pool

"""Thin Python binding of libwf's C ABI (include/wf.h).

Argument marshalling only: every step of the attention path runs in the CUDA
kernels of libwf.so.  Functions keep the C names and take torch CUDA tensors
(or raw integers for pointers).  There is no fallback: if libwf.so is missing
or cannot be loaded, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libwf.so")

WF_OK, WF_ERR_INVALID_ARG, WF_ERR_UNSUPPORTED, WF_ERR_WORKSPACE, WF_ERR_CUDA, WF_ERR_NO_BLOCKS = range(6)
WF_DTYPE_F32, WF_DTYPE_BF16, WF_DTYPE_FP8_E4M3 = 0, 1, 2
WF_DEV_BAD_SLOT, WF_DEV_BAD_BLOCK, WF_DEV_BAD_SEQLEN, WF_DEV_TIMEOUT, WF_DEV_BAD_TASK = 0x1, 0x2, 0x4, 0x8, 0x10
WF_KERNEL_NONE, WF_KERNEL_CUDA_CORES, WF_KERNEL_TENSOR_CORES, WF_KERNEL_TENSOR_CORES_SIMPLE = range(4)

# every entry point include/*.h declares
EXPORTS = (
    "wf_reshape_and_cache",
    "wf_copy_blocks",
    "wf_paged_decode_workspace_size",
    "wf_paged_decode",
    "wf_paged_prefill",
    "wf_paged_prefill_decode",
    "wf_paged_prefill_decode_fused",
    "wf_paged_decode_static_scratch",
    "wf_decode_worker",
    "wf_paged_decode_kernel",
    "wf_paged_prefill_kernel",
    "wf_paged_prefill_persistent",
    "wf_device_status_fetch",
    "wf_status_string",
    "wf_abi_version",
    "wf_bm_create",
    "wf_bm_destroy",
    "wf_bm_num_free",
    "wf_bm_seq_len",
    "wf_bm_ref_count",
    "wf_bm_append",
    "wf_bm_fork",
    "wf_bm_free",
    "wf_bm_tables",
)


class wf_pool_desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
                ("k_head_scales", ctypes.POINTER(ctypes.c_float)), ("v_head_scales", ctypes.POINTER(ctypes.c_float))]


class WfError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn}: {status_string(code)} (status {code})")


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libwf.so (built by paged_kv_cache_wf_gb300.build); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libwf.so not found at {path}: run paged_kv_cache_wf_gb300.build.build()")
        lib = ctypes.CDLL(path)
        vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        lib.wf_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, wf_pool_desc, vp, vp]
        lib.wf_reshape_and_cache.restype = ctypes.c_int
        lib.wf_copy_blocks.argtypes = [vp, vp, vp, i32, wf_pool_desc, vp, vp]
        lib.wf_copy_blocks.restype = ctypes.c_int
        lib.wf_paged_decode_workspace_size.argtypes = [i32, i32, i32, wf_pool_desc]
        lib.wf_paged_decode_workspace_size.restype = sz
        lib.wf_paged_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, f32, wf_pool_desc,
                                        vp, sz, vp, vp]
        lib.wf_paged_decode.restype = ctypes.c_int
        lib.wf_paged_prefill.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, f32,
                                         wf_pool_desc, vp, vp]
        lib.wf_paged_prefill.restype = ctypes.c_int
        lib.wf_paged_prefill_decode.argtypes = [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, vp, vp, vp, i32, vp, i32,
                                                i32, vp, vp, i32, f32, wf_pool_desc, vp, sz, vp, vp]
        lib.wf_paged_prefill_decode.restype = ctypes.c_int
        lib.wf_paged_prefill_decode_fused.argtypes = [wf_pool_desc, i32]
        lib.wf_paged_prefill_decode_fused.restype = ctypes.c_int
        lib.wf_paged_decode_static_scratch.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, f32,
                                                       wf_pool_desc, vp, vp]
        lib.wf_paged_decode_static_scratch.restype = ctypes.c_int
        lib.wf_decode_worker.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, i32, f32, wf_pool_desc, vp, i32, vp,
                                         i32, ctypes.c_uint64, vp, vp]
        lib.wf_decode_worker.restype = ctypes.c_int
        lib.wf_paged_decode_kernel.argtypes = [wf_pool_desc, i32]
        lib.wf_paged_decode_kernel.restype = ctypes.c_int
        lib.wf_paged_prefill_kernel.argtypes = [wf_pool_desc, i32]
        lib.wf_paged_prefill_kernel.restype = ctypes.c_int
        lib.wf_paged_prefill_persistent.argtypes = [wf_pool_desc, i32, i32, i32]
        lib.wf_paged_prefill_persistent.restype = ctypes.c_int
        lib.wf_device_status_fetch.argtypes = [vp, vp, ctypes.c_int, vp]
        lib.wf_device_status_fetch.restype = ctypes.c_int
        lib.wf_status_string.argtypes = [ctypes.c_int]
        lib.wf_status_string.restype = ctypes.c_char_p
        lib.wf_abi_version.argtypes = []
        lib.wf_abi_version.restype = ctypes.c_int
        u64 = ctypes.c_uint64
        lib.wf_bm_create.argtypes = [i32, i32, u64, ctypes.POINTER(vp)]
        lib.wf_bm_create.restype = ctypes.c_int
        lib.wf_bm_destroy.argtypes = [vp]
        lib.wf_bm_destroy.restype = None
        lib.wf_bm_num_free.argtypes = [vp]
        lib.wf_bm_num_free.restype = i32
        lib.wf_bm_seq_len.argtypes = [vp, i64]
        lib.wf_bm_seq_len.restype = i64
        lib.wf_bm_ref_count.argtypes = [vp, i32]
        lib.wf_bm_ref_count.restype = i32
        lib.wf_bm_append.argtypes = [vp, i64, i32, vp, vp, vp]
        lib.wf_bm_append.restype = ctypes.c_int
        lib.wf_bm_fork.argtypes = [vp, i64, i64]
        lib.wf_bm_fork.restype = ctypes.c_int
        lib.wf_bm_free.argtypes = [vp, i64]
        lib.wf_bm_free.restype = ctypes.c_int
        lib.wf_bm_tables.argtypes = [vp, vp, i32, i32, i32, vp, vp]
        lib.wf_bm_tables.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().wf_status_string(code).decode()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int):
    if rc != WF_OK:
        raise WfError(fn, rc)


def _scale_arg(scale):
    """A number -> (per-tensor value, None); a sequence -> (1.0, host float array)."""
    if isinstance(scale, (int, float)):
        return float(scale), None
    vals = [float(x) for x in scale]
    return 1.0, (ctypes.c_float * len(vals))(*vals)


def pool_desc(k_pool, k_scale=1.0, v_scale=1.0) -> wf_pool_desc:
    """Pool geometry from a [N, P, H_kv, D] float32 / bfloat16 tensor, or a uint8
    tensor of fp8 e4m3 codes with its dequantization scales: a number (per tensor)
    or one scale per KV head."""
    import torch
    N, P, H_kv, D = k_pool.shape
    if k_pool.dtype == torch.float32:
        dt = WF_DTYPE_F32
    elif k_pool.dtype == torch.bfloat16:
        dt = WF_DTYPE_BF16
    elif k_pool.dtype == torch.uint8:
        dt = WF_DTYPE_FP8_E4M3
    else:
        raise TypeError(f"unsupported pool dtype {k_pool.dtype}")
    ks, karr = _scale_arg(k_scale)
    vs, varr = _scale_arg(v_scale)
    for arr in (karr, varr):
        if arr is not None and len(arr) != H_kv:
            raise ValueError(f"per-head scales need one value per KV head ({H_kv}), got {len(arr)}")
    d = wf_pool_desc(N, P, H_kv, D, dt, ks, vs, karr, varr)
    d._keep = (karr, varr)   # the host arrays live as long as the descriptor
    return d


def _contig(*ts):
    for t in ts:
        if t is not None and not isinstance(t, int) and not t.is_contiguous():
            raise ValueError("libwf takes dense row-major tensors")


# ---------------------------------------------------------------------------
# the C entry points, torch-tensor flavoured
# ---------------------------------------------------------------------------
def wf_reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, dev_status=None, stream=None,
                         k_scale=1.0, v_scale=1.0):
    """Scatter k, v [T, H_kv, D] into k_pool, v_pool [N, P, H_kv, D] via slot_mapping [T] int64
    (uint8 pools: fp8 e4m3 codes of bf16 k, v quantized with k_scale, v_scale)."""
    _contig(k, v, k_pool, v_pool, slot_mapping)
    lib = load()
    rc = lib.wf_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool), _ptr(slot_mapping),
                                  int(slot_mapping.shape[0]), pool_desc(k_pool, k_scale, v_scale),
                                  _ptr(dev_status), _stream(stream))
    _check("wf_reshape_and_cache", rc)


def wf_copy_blocks(k_pool, v_pool, block_pairs, dev_status=None, stream=None, k_scale=1.0,
                   v_scale=1.0):
    """Copy block src to block dst of both pools for every (src, dst) row of block_pairs [n, 2] int32."""
    _contig(k_pool, v_pool, block_pairs)
    lib = load()
    rc = lib.wf_copy_blocks(_ptr(k_pool), _ptr(v_pool), _ptr(block_pairs), int(block_pairs.shape[0]),
                            pool_desc(k_pool, k_scale, v_scale), _ptr(dev_status), _stream(stream))
    _check("wf_copy_blocks", rc)


def wf_paged_decode_workspace_size(B: int, num_q_heads: int, max_seq_len: int, desc: wf_pool_desc) -> int:
    return int(load().wf_paged_decode_workspace_size(B, num_q_heads, max_seq_len, desc))


def wf_paged_decode(out, q, k_pool, v_pool, block_tables, seq_lens, max_seq_len: int, scale: float,
                    workspace, dev_status=None, stream=None, k_scale=1.0, v_scale=1.0):
    """out, q [B, H_q, D]; block_tables [B, M] int32; seq_lens [B] int32; workspace uint8 tensor."""
    _contig(out, q, k_pool, v_pool, block_tables, seq_lens)
    lib = load()
    B, H_q, _ = q.shape
    rc = lib.wf_paged_decode(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                             int(block_tables.shape[1]), _ptr(seq_lens), int(B), int(max_seq_len),
                             int(H_q), float(scale), pool_desc(k_pool, k_scale, v_scale), _ptr(workspace),
                             int(workspace.numel() * workspace.element_size()), _ptr(dev_status),
                             _stream(stream))
    _check("wf_paged_decode", rc)


def wf_paged_prefill(out, q, k_pool, v_pool, block_tables, seq_lens, cu_q_lens, max_q_len: int,
                     max_seq_len: int, scale: float, dev_status=None, stream=None):
    """out, q [T_total, H_q, D] bf16; cu_q_lens [B+1] int32; seq_lens include the new tokens."""
    _contig(out, q, k_pool, v_pool, block_tables, seq_lens, cu_q_lens)
    lib = load()
    T, H_q, _ = q.shape
    B = int(seq_lens.shape[0])
    rc = lib.wf_paged_prefill(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                              int(block_tables.shape[1]), _ptr(seq_lens), _ptr(cu_q_lens), B, int(T),
                              int(max_q_len), int(max_seq_len), int(H_q), float(scale),
                              pool_desc(k_pool), _ptr(dev_status), _stream(stream))
    _check("wf_paged_prefill", rc)


def wf_paged_prefill_decode_fused(desc: wf_pool_desc, num_q_heads: int) -> bool:
    """Whether wf_paged_prefill_decode runs the step in one grid for this geometry."""
    return bool(load().wf_paged_prefill_decode_fused(desc, int(num_q_heads)))


def wf_paged_prefill_decode(pf_out, pf_q, pf_block_tables, pf_seq_lens, cu_q_lens, max_q_len: int,
                            pf_max_seq_len: int, dec_out, dec_q, dec_block_tables, dec_seq_lens, dec_max_seq_len: int,
                            k_pool, v_pool, scale: float, workspace, dev_status=None, stream=None):
    """The step's prefill (as wf_paged_prefill) and decode (as wf_paged_decode) in one call."""
    _contig(pf_out, pf_q, pf_block_tables, pf_seq_lens, cu_q_lens, dec_out, dec_q, dec_block_tables, dec_seq_lens,
            k_pool, v_pool)
    lib = load()
    T, H_q, _ = pf_q.shape
    rc = lib.wf_paged_prefill_decode(
        _ptr(pf_out), _ptr(pf_q), _ptr(pf_block_tables), int(pf_block_tables.shape[1]), _ptr(pf_seq_lens),
        _ptr(cu_q_lens), int(pf_seq_lens.shape[0]), int(T), int(max_q_len), int(pf_max_seq_len), _ptr(dec_out),
        _ptr(dec_q), _ptr(dec_block_tables), int(dec_block_tables.shape[1]), _ptr(dec_seq_lens),
        int(dec_q.shape[0]), int(dec_max_seq_len), _ptr(k_pool), _ptr(v_pool), int(H_q), float(scale),
        pool_desc(k_pool), _ptr(workspace), int(workspace.numel() * workspace.element_size()), _ptr(dev_status),
        _stream(stream))
    _check("wf_paged_prefill_decode", rc)


WF_STATIC_SCRATCH_BYTES = 32 * 1024 * 1024


def wf_paged_decode_static_scratch(out, q, k_pool, v_pool, block_tables, seq_lens, max_seq_len: int,
                                   scale: float, dev_status=None, stream=None):
    """wf_paged_decode without a caller workspace, for callers that cannot allocate
    device memory: the library's fixed device array is the scratch.  Calls on one
    device share that array, so they must not overlap in time."""
    _contig(out, q, k_pool, v_pool, block_tables, seq_lens)
    lib = load()
    B, H_q, _ = q.shape
    rc = lib.wf_paged_decode_static_scratch(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                            int(block_tables.shape[1]), _ptr(seq_lens), int(B), int(max_seq_len),
                                            int(H_q), float(scale), pool_desc(k_pool), _ptr(dev_status),
                                            _stream(stream))
    _check("wf_paged_decode_static_scratch", rc)


def wf_decode_worker(out, q, k_pool, v_pool, block_tables, tasks, mailbox, scale: float, num_workers: int,
                     idle_timeout_ns: int, dev_status=None, stream=None):
    """Launch the persistent decode worker (returns at once; the grid runs until the
    feeder sets stop or a CTA idles past idle_timeout_ns).  out, q [rows, H_q, D];
    block_tables [table_rows, M] int32; tasks [capacity, 4] int32 records
    (seq_len, table_row, q_row, out_row); mailbox [4] 32-bit words (posted, stop,
    claimed, done), all on the device."""
    _contig(out, q, k_pool, v_pool, block_tables, tasks, mailbox)
    if tasks.dim() != 2 or tasks.shape[1] != 4 or mailbox.numel() != 4:
        raise ValueError("tasks must be [capacity, 4] int32 and mailbox 4 words")
    lib = load()
    rows, H_q, _ = q.shape
    rc = lib.wf_decode_worker(_ptr(out), _ptr(q), int(rows), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                              int(block_tables.shape[0]), int(block_tables.shape[1]), int(H_q), float(scale),
                              pool_desc(k_pool), _ptr(tasks), int(tasks.shape[0]), _ptr(mailbox), int(num_workers),
                              int(idle_timeout_ns), _ptr(dev_status), _stream(stream))
    _check("wf_decode_worker", rc)


def wf_paged_decode_kernel(desc: wf_pool_desc, num_q_heads: int) -> int:
    """The WF_KERNEL_* value of the kernel wf_paged_decode runs for this geometry."""
    return int(load().wf_paged_decode_kernel(desc, int(num_q_heads)))


def wf_paged_prefill_kernel(desc: wf_pool_desc, num_q_heads: int) -> int:
    """The WF_KERNEL_* value of the kernel wf_paged_prefill runs for this geometry."""
    return int(load().wf_paged_prefill_kernel(desc, int(num_q_heads)))


def wf_paged_prefill_persistent(desc: wf_pool_desc, num_q_heads: int, B: int, max_q_len: int) -> bool:
    """Whether wf_paged_prefill runs a batch of this shape as its persistent grid."""
    return bool(load().wf_paged_prefill_persistent(desc, int(num_q_heads), int(B), int(max_q_len)))


def wf_device_status_fetch(dev_status, clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return (optionally clearing) the device status word."""
    lib = load()
    host = ctypes.c_uint32(0)
    rc = lib.wf_device_status_fetch(_ptr(dev_status), ctypes.addressof(host), int(bool(clear)),
                                    _stream(stream))
    _check("wf_device_status_fetch", rc)
    return int(host.value)


# ---------------------------------------------------------------------------
# host-side block manager (include/wf_blocks.h)
# ---------------------------------------------------------------------------
class BlockManager:
    """Blocks of one pool handed out to growing sequences, with reference-counted
    prefix sharing and copy-on-write of shared, partly filled blocks."""

    def __init__(self, num_blocks: int, block_size: int, shuffle_seed: int = 0):
        import numpy as np
        self._np = np
        self.lib = load()
        h = ctypes.c_void_p()
        _check("wf_bm_create", self.lib.wf_bm_create(int(num_blocks), int(block_size), int(shuffle_seed),
                                                      ctypes.byref(h)))
        self.h = h
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if self.h:
            self.lib.wf_bm_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return int(self.lib.wf_bm_num_free(self.h))

    def seq_len(self, seq: int) -> int:
        return int(self.lib.wf_bm_seq_len(self.h, int(seq)))

    def ref_count(self, block: int) -> int:
        return int(self.lib.wf_bm_ref_count(self.h, int(block)))

    def append(self, seq: int, n: int):
        """Slots (int64 [n]) of n new tokens of `seq`, and the copy-on-write pair
        (src, dst) to copy before writing them, or None."""
        np = self._np
        slots = np.zeros(max(int(n), 1), np.int64)
        pair = np.zeros(2, np.int32)
        ncow = ctypes.c_int32(0)
        _check("wf_bm_append", self.lib.wf_bm_append(self.h, int(seq), int(n), slots.ctypes.data,
                                                      pair.ctypes.data, ctypes.byref(ncow)))
        return slots[:int(n)], (tuple(int(x) for x in pair) if ncow.value else None)

    def fork(self, parent: int, child: int):
        _check("wf_bm_fork", self.lib.wf_bm_fork(self.h, int(parent), int(child)))

    def free(self, seq: int):
        _check("wf_bm_free", self.lib.wf_bm_free(self.h, int(seq)))

    def tables(self, seqs, M: int, pad_block: int):
        """block_tables int32 [B, M] and seq_lens int32 [B] of the sequences `seqs`."""
        np = self._np
        ids = np.ascontiguousarray(np.asarray(seqs, np.int64))
        B = int(ids.shape[0])
        bt = np.zeros((max(B, 1), int(M)), np.int32)
        sl = np.zeros(max(B, 1), np.int32)
        _check("wf_bm_tables", self.lib.wf_bm_tables(self.h, ids.ctypes.data, B, int(M), int(pad_block),
                                                      bt.ctypes.data, sl.ctypes.data))
        return bt[:B], sl[:B]

"""GB300 (sm_103a) paged-KV attention: Python binding of the C-ABI library.

Functions here carry the C entry points' names (``include/pa.h``) and only
marshal arguments: every step of the path runs in the library's CUDA kernels.
There is no CPU fallback: if ``libpa_gb300.so`` has not been built, or CUDA is
unavailable, calls raise.

Build the library with ``paged_kv_cache_240_gb300._build.build()`` (or the repo's
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "PaError", "PagedCache", "load_library", "pa_write_kv", "pa_decode",
    "pa_decode_partitioned", "pa_decode_workspace_bytes", "pa_decode_noalloc",
    "pa_decode_append", "pa_prefill_chunk",
    "pa_status_str", "pa_check_flags", "PA_FLAG_SLOT_RANGE", "PA_FLAG_BLOCK_ID",
    "PA_FLAG_CONTEXT_LEN", "PA_FLAG_Q_LEN", "PA_FLAG_TIMEOUT", "EXPORTED_SYMBOLS",
    "pa_last_cuda_error", "pa_selftest_bounded_wait",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa_gb300.so")

(PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_DEVICE_DATA,
 PA_ERR_OUT_OF_BLOCKS) = range(6)
PA_F16, PA_BF16, PA_I8 = 0, 1, 2
PA_FLAG_SLOT_RANGE, PA_FLAG_BLOCK_ID, PA_FLAG_CONTEXT_LEN, PA_FLAG_Q_LEN, PA_FLAG_TIMEOUT = (
    1, 2, 4, 8, 16)

EXPORTED_SYMBOLS = ("pa_write_kv", "pa_decode", "pa_decode_partitioned",
                    "pa_decode_workspace_bytes", "pa_decode_noalloc", "pa_decode_append",
                    "pa_prefill_chunk",
                    "pa_status_str", "pa_last_cuda_error", "pa_check_flags",
                    "pa_blocks_create", "pa_blocks_destroy", "pa_blocks_append",
                    "pa_blocks_rollback", "pa_blocks_release", "pa_blocks_preempt",
                    "pa_blocks_evict_window", "pa_blocks_tables", "pa_blocks_context_len",
                    "pa_blocks_get_stats", "pa_blocks_publish", "pa_blocks_attach_prefix",
                    "pa_linear_int8_quantize", "pa_linear_int8_workspace_bytes",
                    "pa_linear_int8", "pa_linear_int8_grouped", "pa_selftest_bounded_wait")
PA_NOALLOC_SCRATCH_BYTES = 16 << 20


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s" % (what, _status_name(status)))


class _PaCacheStruct(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("dtype", ctypes.c_int), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it was not built)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("CUDA library %s is not built; run "
                           "paged_kv_cache_240_gb300._build.build()" % path)
    lib = ctypes.CDLL(path)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    cp = ctypes.POINTER(_PaCacheStruct)
    lib.pa_write_kv.argtypes = [cp, P, P, I, P, I, P, P]
    lib.pa_decode.argtypes = [cp, P, P, I, I, I, P, I, P, F, I, P, S, P, P]
    lib.pa_decode_partitioned.argtypes = [cp, P, P, I, I, I, P, I, P, F, I, I, P, S, P, P]
    lib.pa_decode_noalloc.argtypes = [cp, P, P, I, I, I, P, I, P, F, I, P, P]
    lib.pa_decode_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    lib.pa_decode_workspace_bytes.restype = S
    lib.pa_prefill_chunk.argtypes = [cp, P, P, I, I, I, I, P, I, P, I, P, F, I, P, S, P, P]
    lib.pa_status_str.argtypes = [I]
    lib.pa_status_str.restype = ctypes.c_char_p
    lib.pa_check_flags.argtypes = [ctypes.c_int32]
    lib.pa_last_cuda_error.argtypes = []
    lib.pa_last_cuda_error.restype = ctypes.c_char_p
    lib.pa_selftest_bounded_wait.argtypes = [ctypes.c_longlong, P, P, P]
    lib.pa_decode_append.argtypes = [cp, P, P, I, P, P, I, I, I, P, I, P, F, I, P, S, P, P]
    for name in ("pa_write_kv", "pa_decode", "pa_decode_partitioned", "pa_decode_noalloc",
                 "pa_decode_append", "pa_prefill_chunk", "pa_check_flags",
                 "pa_selftest_bounded_wait"):
        getattr(lib, name).restype = I
    if path == LIB_PATH:
        _lib = lib
    return lib


def _status_name(status: int) -> str:
    try:
        return load_library().pa_status_str(status).decode()
    except Exception:  # library missing: still say which code it was
        return "status %d" % status


def pa_status_str(status: int) -> str:
    return load_library().pa_status_str(int(status)).decode()


def pa_last_cuda_error() -> str:
    """Text of the CUDA error behind this thread's most recent PA_ERR_CUDA."""
    return load_library().pa_last_cuda_error().decode()


def pa_check_flags(flags: int) -> int:
    return load_library().pa_check_flags(int(flags))


# ------------------------------------------------------------------ tensors

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.int8:
        return PA_I8
    raise ValueError("unsupported dtype %s" % t.dtype)


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensor must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")


def _raise(status: int, what: str):
    if status == PA_ERR_CUDA:
        raise PaError(status, "%s (%s)" % (what, load_library().pa_last_cuda_error().decode()))
    if status != PA_OK:
        raise PaError(status, what)


class PagedCache:
    """A paged KV cache in device memory.

    ``k``/``v``: [num_blocks, num_kv_heads, 16, head_dim] of float16, bfloat16 or
    int8; int8 caches also hold ``k_scale``/``v_scale`` [num_blocks, num_kv_heads,
    16] float32.  The tensors may be given (then they are used as they are) or
    are allocated (uninitialised)."""

    def __init__(self, num_blocks: int, num_kv_heads: int, head_dim: int, dtype,
                 device="cuda", k=None, v=None, k_scale=None, v_scale=None,
                 block_size: int = 16):
        torch = _torch()
        dt = {"f16": torch.float16, "bf16": torch.bfloat16, "i8": torch.int8}.get(dtype, dtype)
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        self.k = k if k is not None else torch.empty(shape, dtype=dt, device=device)
        self.v = v if v is not None else torch.empty(shape, dtype=dt, device=device)
        self.k_scale = self.v_scale = None
        if dt == torch.int8:
            self.k_scale = k_scale if k_scale is not None else torch.empty(
                shape[:3], dtype=torch.float32, device=device)
            self.v_scale = v_scale if v_scale is not None else torch.empty(
                shape[:3], dtype=torch.float32, device=device)
        for t in (self.k, self.v):
            if tuple(t.shape) != shape or t.dtype != dt:
                raise ValueError("cache tensor has shape %s / %s, expected %s / %s"
                                 % (tuple(t.shape), t.dtype, shape, dt))
        _check_cuda(self.k, self.v, self.k_scale, self.v_scale)
        self.num_blocks, self.num_kv_heads, self.head_dim = num_blocks, num_kv_heads, head_dim
        self.block_size = block_size
        self.dtype_code = _dtype_code(self.k)

    def struct(self) -> _PaCacheStruct:
        return _PaCacheStruct(self.num_blocks, self.block_size, self.num_kv_heads,
                              self.head_dim, self.dtype_code, self.k.data_ptr(),
                              self.v.data_ptr(),
                              None if self.k_scale is None else self.k_scale.data_ptr(),
                              None if self.v_scale is None else self.v_scale.data_ptr())


def pa_write_kv(cache: PagedCache, k, v, slot_mapping, err_flag, stream=None):
    """Scatter rows k, v [T, Hkv, D] into their slots (int8 caches quantise)."""
    _check_cuda(k, v, slot_mapping, err_flag)
    st = cache.struct()
    _raise(load_library().pa_write_kv(ctypes.byref(st), _ptr(k), _ptr(v), _dtype_code(k),
                                      _ptr(slot_mapping), int(slot_mapping.shape[0]),
                                      _ptr(err_flag), _stream(stream)), "pa_write_kv")


def pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                              max_blocks_per_seq, window=0, partition_blocks=0) -> int:
    n = load_library().pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 max_blocks_per_seq, window, partition_blocks)
    if n == ctypes.c_size_t(-1).value:
        raise PaError(PA_ERR_INVALID_ARG, "pa_decode_workspace_bytes")
    return n


def pa_decode_partitioned(cache: PagedCache, out, q, block_tables, context_lens, sm_scale,
                          window, partition_blocks, workspace, err_flag, stream=None):
    _check_cuda(out, q, block_tables, context_lens, workspace, err_flag)
    st = cache.struct()
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _raise(load_library().pa_decode_partitioned(
        ctypes.byref(st), _ptr(out), _ptr(q), _dtype_code(q), int(q.shape[0]), int(q.shape[1]),
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), float(sm_scale),
        int(window), int(partition_blocks), _ptr(workspace), nbytes, _ptr(err_flag),
        _stream(stream)), "pa_decode")


def pa_decode(cache: PagedCache, out, q, block_tables, context_lens, sm_scale, window,
              workspace, err_flag, stream=None):
    """q, out [B, Hq, D]; block_tables [B, MB] int32; context_lens [B] int32."""
    _check_cuda(out, q, block_tables, context_lens, workspace, err_flag)
    st = cache.struct()
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _raise(load_library().pa_decode(
        ctypes.byref(st), _ptr(out), _ptr(q), _dtype_code(q), int(q.shape[0]), int(q.shape[1]),
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), float(sm_scale),
        int(window), _ptr(workspace), nbytes, _ptr(err_flag), _stream(stream)), "pa_decode")


def pa_decode_append(cache: PagedCache, k_new, v_new, out, q, block_tables, context_lens,
                     sm_scale, window, workspace, err_flag, stream=None):
    """One decode step in one launch: k_new, v_new [B, Hkv, D] written at each
    sequence's position context_lens[b] - 1, then q, out [B, Hq, D] attend; the
    same bits as pa_write_kv of those slots followed by pa_decode."""
    _check_cuda(k_new, v_new, out, q, block_tables, context_lens, workspace, err_flag)
    st = cache.struct()
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _raise(load_library().pa_decode_append(
        ctypes.byref(st), _ptr(k_new), _ptr(v_new), _dtype_code(k_new), _ptr(out), _ptr(q),
        _dtype_code(q), int(q.shape[0]), int(q.shape[1]), _ptr(block_tables),
        int(block_tables.shape[1]), _ptr(context_lens), float(sm_scale), int(window),
        _ptr(workspace), nbytes, _ptr(err_flag), _stream(stream)), "pa_decode_append")


def pa_decode_noalloc(cache: PagedCache, out, q, block_tables, context_lens, sm_scale, window,
                      err_flag, stream=None):
    """pa_decode for callers that cannot allocate device memory: the split-K
    partials use scratch compiled into the library (PA_NOALLOC_SCRATCH_BYTES per
    device).  Raises PaError (PA_ERR_UNSUPPORTED) when a batch needs more."""
    _check_cuda(out, q, block_tables, context_lens, err_flag)
    st = cache.struct()
    _raise(load_library().pa_decode_noalloc(
        ctypes.byref(st), _ptr(out), _ptr(q), _dtype_code(q), int(q.shape[0]), int(q.shape[1]),
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), float(sm_scale),
        int(window), _ptr(err_flag), _stream(stream)), "pa_decode_noalloc")


def pa_prefill_chunk(cache: PagedCache, out, q, cu_q_lens, max_q_len, block_tables,
                     context_lens, sm_scale, window, err_flag, stream=None):
    """q, out [T, Hq, D]; cu_q_lens [n+1] int32; block_tables [n, MB]; context_lens [n]."""
    _check_cuda(out, q, cu_q_lens, block_tables, context_lens, err_flag)
    st = cache.struct()
    _raise(load_library().pa_prefill_chunk(
        ctypes.byref(st), _ptr(out), _ptr(q), _dtype_code(q), int(q.shape[0]),
        int(cu_q_lens.shape[0]) - 1, int(q.shape[1]), _ptr(cu_q_lens), int(max_q_len),
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), float(sm_scale),
        int(window), None, 0, _ptr(err_flag), _stream(stream)), "pa_prefill_chunk")


def pa_selftest_bounded_wait(limit_cycles, result, err_flag, stream=None):
    """Run the bounded-wait self-check: result is a device int64 tensor [4]."""
    _check_cuda(result, err_flag)
    _raise(load_library().pa_selftest_bounded_wait(int(limit_cycles), _ptr(result),
                                                   _ptr(err_flag), _stream(stream)),
           "pa_selftest_bounded_wait")

"""CPU oracle for attention over a paged KV cache -- TEST INFRASTRUCTURE ONLY.

This package wraps ``pa_oracle.c`` (plain C, fp64 attention, fp32 IEEE int8
quantisation) through ctypes.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import it.  The CUDA library
in ``paged_kv_cache_240_gb300`` never imports, links or calls it, and the two
share no code.

Every array argument is a numpy array in the layout the C file documents:
caches ``[num_blocks, num_kv_heads, block_size, head_dim]`` (16-bit caches as
uint16 bit patterns, int8 caches as int8 codes), scales
``[num_blocks, num_kv_heads, block_size]`` float32, q ``[tokens, q_heads,
head_dim]`` uint16 bits, block tables ``[seqs, max_blocks_per_seq]`` int32.

What each function computes, and the page passages it follows, is stated in the
C source beside the function.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")

DTYPES = {"f16": 0, "bf16": 1, "i8": 2}

# Plain IEEE arithmetic: no fused multiply-add contraction, no fast-math.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-frounding-math"]


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc into a shared library (idempotent)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


_lib_cache: dict[str, ctypes.CDLL] = {}


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library; ``path`` selects
    another build of the same source (the mutation tests use this)."""
    path = path or build()
    if path in _lib_cache:
        return _lib_cache[path]
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.pao_f16_to_double.restype = ctypes.c_double
    lib.pao_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.pao_bf16_to_double.restype = ctypes.c_double
    lib.pao_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.pao_quantize_row.restype = None
    lib.pao_quantize_row.argtypes = [P, i, P, P]
    lib.pao_write_kv.restype = i
    lib.pao_write_kv.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, P, i]
    att = [i, i, i, i, i, P, P, P, P, i, P, i, i, P, P, i, P, ctypes.c_double, i]
    lib.pao_attention.restype = i
    lib.pao_attention.argtypes = att + [P]
    lib.pao_attention_online.restype = i
    lib.pao_attention_online.argtypes = att + [i, P, i, P]
    lib.pao_quantize_weights.argtypes = [i, P, i, i, P, P]
    lib.pao_quantize_weights.restype = None
    lib.pao_linear_int8.argtypes = [P, P, i, P, i, P, i, i, i, P]
    lib.pao_linear_int8.restype = None
    _lib_cache[path] = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def f16_to_double(bits: int, lib=None) -> float:
    return (lib or load()).pao_f16_to_double(int(bits))


def bf16_to_double(bits: int, lib=None) -> float:
    return (lib or load()).pao_bf16_to_double(int(bits))


def quantize_row(x, lib=None):
    """int8 codes and fp32 scale of one row (see ``pao_quantize_row``)."""
    x = _c(x, np.float32)
    codes = np.zeros(x.shape[0], np.int8)
    scale = np.zeros(1, np.float32)
    (lib or load()).pao_quantize_row(_ptr(x), x.shape[0], _ptr(codes), _ptr(scale))
    return codes, scale[0]


class Cache:
    """A paged KV cache held in host memory (numpy), as the oracle sees it."""

    def __init__(self, dtype: str, num_blocks: int, num_kv_heads: int, head_dim: int,
                 block_size: int = 16, k=None, v=None, k_scale=None, v_scale=None):
        self.dtype = dtype
        self.num_blocks, self.num_kv_heads = num_blocks, num_kv_heads
        self.head_dim, self.block_size = head_dim, block_size
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        el = np.int8 if dtype == "i8" else np.uint16
        self.k = _c(k, el) if k is not None else np.zeros(shape, el)
        self.v = _c(v, el) if v is not None else np.zeros(shape, el)
        if dtype == "i8":
            sshape = shape[:3]
            self.k_scale = _c(k_scale, np.float32) if k_scale is not None else np.zeros(sshape, np.float32)
            self.v_scale = _c(v_scale, np.float32) if v_scale is not None else np.zeros(sshape, np.float32)
        else:
            self.k_scale = self.v_scale = None
        assert self.k.shape == shape and self.v.shape == shape

    def copy(self) -> "Cache":
        return Cache(self.dtype, self.num_blocks, self.num_kv_heads, self.head_dim,
                     self.block_size, self.k.copy(), self.v.copy(),
                     None if self.k_scale is None else self.k_scale.copy(),
                     None if self.v_scale is None else self.v_scale.copy())


def write_kv(cache: Cache, k_bits, v_bits, in_dtype: str, slot_mapping, lib=None) -> int:
    """Write new tokens' K/V rows (uint16 bits, [T, Hkv, D]) into ``cache`` in
    place.  Returns the number of out-of-range slots that were skipped."""
    k_bits, v_bits = _c(k_bits, np.uint16), _c(v_bits, np.uint16)
    slot_mapping = _c(slot_mapping, np.int32)
    T = slot_mapping.shape[0]
    assert k_bits.shape == (T, cache.num_kv_heads, cache.head_dim) == v_bits.shape
    return (lib or load()).pao_write_kv(
        DTYPES[cache.dtype], DTYPES[in_dtype], cache.num_blocks, cache.block_size,
        cache.num_kv_heads, cache.head_dim, _ptr(cache.k), _ptr(cache.v),
        _ptr(cache.k_scale), _ptr(cache.v_scale), _ptr(k_bits), _ptr(v_bits),
        _ptr(slot_mapping), T)


def _att_args(cache, q_bits, q_dtype, cu_q_lens, block_tables, context_lens, sm_scale, window):
    q_bits = _c(q_bits, np.uint16)
    cu_q_lens = _c(cu_q_lens, np.int32)
    block_tables = _c(block_tables, np.int32)
    context_lens = _c(context_lens, np.int32)
    T, Hq, D = q_bits.shape
    assert D == cache.head_dim and Hq % cache.num_kv_heads == 0
    B = context_lens.shape[0]
    assert cu_q_lens.shape == (B + 1,) and cu_q_lens[-1] == T
    assert block_tables.shape[0] == B
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    keep = (q_bits, cu_q_lens, block_tables, context_lens)
    args = [DTYPES[cache.dtype], cache.num_blocks, cache.block_size, cache.num_kv_heads,
            cache.head_dim, _ptr(cache.k), _ptr(cache.v), _ptr(cache.k_scale),
            _ptr(cache.v_scale), DTYPES[q_dtype], _ptr(q_bits), B, Hq, _ptr(cu_q_lens),
            _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            float(sm_scale), int(window)]
    return args, keep, (T, Hq, D)


def attention(cache: Cache, q_bits, q_dtype, cu_q_lens, block_tables, context_lens,
              sm_scale=None, window=0, lib=None) -> np.ndarray:
    """fp64 attention over the paged cache by its definition (two-pass softmax).
    ``sm_scale`` defaults to 1/sqrt(head_dim).  Returns [T, Hq, D] float64."""
    args, keep, shape = _att_args(cache, q_bits, q_dtype, cu_q_lens, block_tables,
                                  context_lens, sm_scale, window)
    out = np.zeros(shape, np.float64)
    (lib or load()).pao_attention(*args, _ptr(out))
    return out


def attention_online(cache: Cache, q_bits, q_dtype, cu_q_lens, block_tables,
                     context_lens, sm_scale=None, window=0, part_tokens=256,
                     seg_lens=(16,), lib=None) -> np.ndarray:
    """fp64 attention reached by the online-softmax walk over segments and a
    split-K merge of partitions of ``part_tokens`` keys."""
    args, keep, shape = _att_args(cache, q_bits, q_dtype, cu_q_lens, block_tables,
                                  context_lens, sm_scale, window)
    seg = _c(seg_lens, np.int32)
    assert seg.size > 0 and (seg > 0).all() and part_tokens > 0
    out = np.zeros(shape, np.float64)
    (lib or load()).pao_attention_online(*args, int(part_tokens), _ptr(seg), seg.size,
                                         _ptr(out))
    return out


def quantize_weights(w_bits, w_dtype: str, lib=None):
    """Per-output-channel int8 codes [n, k] and fp32 scales [n] of w [n, k]
    (16-bit bit patterns); see ``pao_quantize_weights``."""
    w = _c(w_bits, np.uint16)
    n, k = w.shape
    codes = np.zeros((n, k), np.int8)
    scales = np.zeros(n, np.float32)
    (lib or load()).pao_quantize_weights(DTYPES[w_dtype], _ptr(w), n, k, _ptr(codes),
                                         _ptr(scales))
    return codes, scales


def linear_int8(codes, scales, x_bits, x_dtype: str, bias_bits=None, lib=None):
    """y [m, n] (fp64) = x * (codes * scales)^T (+ bias); see ``pao_linear_int8``."""
    codes = _c(codes, np.int8)
    scales = _c(scales, np.float32)
    x = _c(x_bits, np.uint16)
    m, k = x.shape
    n = codes.shape[0]
    assert codes.shape == (n, k) and scales.shape == (n,)
    y = np.zeros((m, n), np.float64)
    bias = _c(bias_bits, np.uint16) if bias_bits is not None else np.zeros(1, np.uint16)
    (lib or load()).pao_linear_int8(_ptr(codes), _ptr(scales), DTYPES[x_dtype], _ptr(x),
                                    int(bias_bits is not None), _ptr(bias), m, n, k, _ptr(y))
    return y


def decode_cu_q_lens(num_seqs: int) -> np.ndarray:
    """cu_q_lens of a decode batch: one query per sequence."""
    return np.arange(num_seqs + 1, dtype=np.int32)

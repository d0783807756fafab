"""The C-ABI library builds, loads and exports every entry point include/pa.h,
include/pa_blocks.h and include/pa_linear.h declare; host-side argument checks reject bad calls before any launch (no GPU
needed: these calls never reach CUDA)."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_cache_240_gb300 as pa
from paged_kv_cache_240_gb300 import _build

HEADERS = [os.path.join(_build.INCLUDE, h) for h in ("pa.h", "pa_blocks.h", "pa_linear.h")]


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pa.load_library()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_matches_binding():
    assert declared_functions() == sorted(pa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pa_[a-z0-9_]+)\b", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    assert pa.pa_status_str(0) == "PA_OK"
    assert pa.pa_status_str(4) == "PA_ERR_DEVICE_DATA"
    assert pa.pa_check_flags(0) == 0
    assert pa.pa_check_flags(pa.PA_FLAG_BLOCK_ID) == 4
    assert pa.pa_last_cuda_error() == "no CUDA error"  # nothing has failed on this thread


def _cache(**kw):
    f = dict(num_blocks=4, block_size=16, num_kv_heads=2, head_dim=128, dtype=0,
             k_cache=4096, v_cache=8192, k_scale=None, v_scale=None)
    f.update(kw)
    return pa._PaCacheStruct(**f)


def test_write_rejects_bad_arguments(lib):
    err = ctypes.c_void_p(16 * 99)
    call = lambda c, **kw: lib.pa_write_kv(ctypes.byref(c), kw.get("k", 256), kw.get("v", 512),
                                           kw.get("dt", 0), kw.get("slots", 768),
                                           kw.get("n", 3), kw.get("err", err), None)
    assert lib.pa_write_kv(None, 1, 1, 0, 1, 1, err, None) == pa.PA_ERR_INVALID_ARG
    assert call(_cache(block_size=8)) == pa.PA_ERR_UNSUPPORTED
    assert call(_cache(head_dim=96)) == pa.PA_ERR_UNSUPPORTED
    assert call(_cache(dtype=7)) == pa.PA_ERR_UNSUPPORTED
    assert call(_cache(k_cache=None)) == pa.PA_ERR_INVALID_ARG
    assert call(_cache(k_cache=4100)) == pa.PA_ERR_INVALID_ARG          # misaligned
    assert call(_cache(dtype=2)) == pa.PA_ERR_INVALID_ARG               # int8 without scales
    assert call(_cache(), dt=1) == pa.PA_ERR_UNSUPPORTED                # bf16 into f16 cache
    assert call(_cache(), n=-1) == pa.PA_ERR_INVALID_ARG
    assert call(_cache(), err=None) == pa.PA_ERR_INVALID_ARG
    assert call(_cache(), n=0) == pa.PA_OK                              # no-op, nothing launched


def test_decode_rejects_bad_arguments(lib):
    err = ctypes.c_void_p(16 * 99)

    def call(c, **kw):
        return lib.pa_decode(ctypes.byref(c), 256, 512, kw.get("qdt", 0), kw.get("B", 2),
                             kw.get("Hq", 4), 768, kw.get("MB", 4), 1024, kw.get("sm", 0.1),
                             kw.get("W", 0), None, 0, kw.get("err", err), None)
    assert call(_cache(), Hq=3) == pa.PA_ERR_INVALID_ARG       # Hq % Hkv != 0
    assert call(_cache(), qdt=1) == pa.PA_ERR_UNSUPPORTED      # q type != cache type
    assert call(_cache(), MB=0) == pa.PA_ERR_INVALID_ARG
    assert call(_cache(), W=-1) == pa.PA_ERR_INVALID_ARG
    assert call(_cache(), sm=float("nan")) == pa.PA_ERR_INVALID_ARG
    assert call(_cache(), B=0) == pa.PA_OK
    assert lib.pa_decode_workspace_bytes(2, 3, 2, 128, 4, 0, 0) == ctypes.c_size_t(-1).value
    assert lib.pa_decode_workspace_bytes(2, 4, 2, 96, 4, 0, 0) == ctypes.c_size_t(-1).value


def test_decode_append_rejects_bad_arguments(lib):
    err = ctypes.c_void_p(16 * 99)

    def call(c, **kw):
        return lib.pa_decode_append(ctypes.byref(c), kw.get("k", 1280), kw.get("v", 1536),
                                    kw.get("kvdt", 0), 256, 512, kw.get("qdt", 0),
                                    kw.get("B", 2), kw.get("Hq", 4), 768, 4, 1024, 0.1, 0, None,
                                    0, kw.get("err", err), None)
    assert call(_cache(), Hq=3) == pa.PA_ERR_INVALID_ARG       # Hq % Hkv != 0
    assert call(_cache(), qdt=1) == pa.PA_ERR_UNSUPPORTED      # q type != cache type
    assert call(_cache(), k=None) == pa.PA_ERR_INVALID_ARG     # no new K rows
    assert call(_cache(), v=1544) == pa.PA_ERR_INVALID_ARG     # misaligned new V rows
    assert call(_cache(), kvdt=1) == pa.PA_ERR_UNSUPPORTED     # new rows' type != q's
    assert call(_cache(), err=None) == pa.PA_ERR_INVALID_ARG
    assert call(_cache(), B=0) == pa.PA_OK


def test_prefill_rejects_bad_arguments(lib):
    err = ctypes.c_void_p(16 * 99)

    def call(c, **kw):
        return lib.pa_prefill_chunk(ctypes.byref(c), 256, 512, kw.get("qdt", 0), kw.get("T", 8),
                                    kw.get("n", 2), kw.get("Hq", 4), 768, kw.get("mq", 4), 1024,
                                    4, 1280, 0.1, 0, None, 0, kw.get("err", err), None)
    assert call(_cache(), Hq=5) == pa.PA_ERR_INVALID_ARG
    assert call(_cache(), mq=-1) == pa.PA_ERR_INVALID_ARG
    assert call(_cache(), qdt=2) == pa.PA_ERR_UNSUPPORTED
    assert call(_cache(), T=0) == pa.PA_OK


def test_linear_rejects_bad_arguments():
    """include/pa_linear.h: the host checks return before any launch (fake,
    never dereferenced addresses; 16-byte aligned unless the case says not)."""
    from paged_kv_cache_240_gb300 import linear as L
    lib = L._lib()
    A = 1 << 20  # an aligned fake address

    def lin(codes=A, scales=A, x=A, y=A, xdt=pa.PA_BF16, m=8, n=64, k=256, ws=None):
        return lib.pa_linear_int8(codes, scales, None, x, xdt, m, n, k, y, ws, 0, None)

    assert lin(codes=None) == pa.PA_ERR_INVALID_ARG
    assert lin(x=None) == pa.PA_ERR_INVALID_ARG
    assert lin(m=0) == pa.PA_ERR_INVALID_ARG
    assert lin(xdt=pa.PA_I8) == pa.PA_ERR_UNSUPPORTED
    assert lin(n=24) == pa.PA_ERR_UNSUPPORTED          # n % 16
    assert lin(k=96) == pa.PA_ERR_UNSUPPORTED          # k % 64
    assert lin(k=65536 + 64) == pa.PA_ERR_UNSUPPORTED  # k too large
    assert lin(codes=A + 8) == pa.PA_ERR_INVALID_ARG   # codes not 16-byte aligned
    assert lin(x=A + 4) == pa.PA_ERR_INVALID_ARG       # x not 16-byte aligned
    assert lin(y=A + 1) == pa.PA_ERR_INVALID_ARG       # y not 2-byte aligned
    assert lin(scales=A + 2) == pa.PA_ERR_INVALID_ARG  # scales not 4-byte aligned

    import ctypes as C
    P4, N4 = C.c_void_p * 4, C.c_int * 4

    def grp(count=2, codes=(A, A), scales=(A, A), n=(64, 32), x=A, y=(A, A), xdt=pa.PA_BF16,
            m=8, k=256):
        return lib.pa_linear_int8_grouped(count, P4(*codes), P4(*scales), None, N4(*n), x, xdt,
                                          m, k, P4(*y), None)

    assert grp(count=0) == pa.PA_ERR_INVALID_ARG
    assert grp(count=5) == pa.PA_ERR_INVALID_ARG
    assert grp(codes=(A, None)) == pa.PA_ERR_INVALID_ARG
    assert grp(n=(64, 24)) == pa.PA_ERR_UNSUPPORTED      # n % 16
    assert grp(k=96) == pa.PA_ERR_UNSUPPORTED            # k % 64
    assert grp(codes=(A, A + 8)) == pa.PA_ERR_INVALID_ARG
    assert grp(y=(A + 1, A)) == pa.PA_ERR_INVALID_ARG
    assert grp(x=A + 4) == pa.PA_ERR_INVALID_ARG
    assert grp(xdt=pa.PA_I8) == pa.PA_ERR_UNSUPPORTED

    q = lib.pa_linear_int8_quantize
    assert q(None, pa.PA_BF16, 16, 64, A, A, None) == pa.PA_ERR_INVALID_ARG
    assert q(A, pa.PA_I8, 16, 64, A, A, None) == pa.PA_ERR_UNSUPPORTED
    assert q(A, pa.PA_F16, 0, 64, A, A, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_linear_int8_workspace_bytes(0, 64, 64) == 0

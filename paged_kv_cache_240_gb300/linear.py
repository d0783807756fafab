"""ctypes binding of include/pa_linear.h: the weight-only INT8 linear layer
(argument marshalling only; the work is the CUDA library's)."""
from __future__ import annotations

import ctypes

from . import (PaError, _check_cuda, _dtype_code, _ptr, _raise, _stream, _torch,
               load_library)


def _lib():
    lib = load_library()
    if not getattr(lib, "_pa_linear_ready", False):
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.pa_linear_int8_quantize.argtypes = [P, I, I, I, P, P, P]
        lib.pa_linear_int8_quantize.restype = I
        lib.pa_linear_int8_workspace_bytes.argtypes = [I, I, I]
        lib.pa_linear_int8_workspace_bytes.restype = S
        lib.pa_linear_int8.argtypes = [P, P, P, P, I, I, I, I, P, P, S, P]
        lib.pa_linear_int8.restype = I
        lib.pa_linear_int8_grouped.argtypes = [I, P, P, P, P, P, I, I, I, P, P]
        lib.pa_linear_int8_grouped.restype = I
        lib._pa_linear_ready = True
    return lib


def int8_quantize(w, codes=None, scales=None, stream=None):
    """w [n, k] fp16/bf16 (CUDA) -> (codes int8 [n, k], scales fp32 [n])."""
    torch = _torch()
    n, k = w.shape
    if codes is None:
        codes = torch.empty((n, k), dtype=torch.int8, device=w.device)
    if scales is None:
        scales = torch.empty(n, dtype=torch.float32, device=w.device)
    _check_cuda(w, codes, scales)
    _raise(_lib().pa_linear_int8_quantize(_ptr(w), _dtype_code(w), n, k, _ptr(codes),
                                          _ptr(scales), _stream(stream)), "pa_linear_int8_quantize")
    return codes, scales


def int8_workspace_bytes(m: int, n: int, k: int) -> int:
    return int(_lib().pa_linear_int8_workspace_bytes(m, n, k))


def int8_linear(codes, scales, x, bias=None, out=None, workspace=None, stream=None):
    """y [m, n] = x [m, k] * dequant(codes, scales)^T (+ bias), in x's dtype."""
    torch = _torch()
    m, k = x.shape
    n = codes.shape[0]
    if codes.shape[1] != k or scales.shape[0] != n:
        raise PaError(1, "pa_linear_int8")
    if out is None:
        out = torch.empty((m, n), dtype=x.dtype, device=x.device)
    _check_cuda(codes, scales, x, bias, out, workspace)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _raise(_lib().pa_linear_int8(_ptr(codes), _ptr(scales), _ptr(bias), _ptr(x),
                                 _dtype_code(x), m, n, k, _ptr(out), _ptr(workspace), nbytes,
                                 _stream(stream)), "pa_linear_int8")
    return out


def int8_linear_grouped(mats, x, outs=None, stream=None):
    """One launch for up to four linears that read the same x [m, k]: mats is a
    list of (codes [n_i, k], scales [n_i], bias [n_i] or None); returns the
    outputs [m, n_i] in x's dtype (or fills ``outs``)."""
    torch = _torch()
    m, k = x.shape
    count = len(mats)
    if not 1 <= count <= 4:
        raise PaError(1, "pa_linear_int8_grouped")
    if outs is None:
        outs = [torch.empty((m, c.shape[0]), dtype=x.dtype, device=x.device) for c, _, _ in mats]
    for (codes, scales, bias), y in zip(mats, outs):
        if codes.shape[1] != k or scales.shape[0] != codes.shape[0]:
            raise PaError(1, "pa_linear_int8_grouped")
        _check_cuda(codes, scales, bias, y)
    _check_cuda(x)
    vp = ctypes.c_void_p * count
    arr_codes = vp(*[c.data_ptr() for c, _, _ in mats])
    arr_scales = vp(*[s.data_ptr() for _, s, _ in mats])
    arr_bias = vp(*[0 if b is None else b.data_ptr() for _, _, b in mats])
    arr_y = vp(*[y.data_ptr() for y in outs])
    arr_n = (ctypes.c_int * count)(*[int(c.shape[0]) for c, _, _ in mats])
    _raise(_lib().pa_linear_int8_grouped(count, arr_codes, arr_scales, arr_bias, arr_n, _ptr(x),
                                         _dtype_code(x), m, k, arr_y, _stream(stream)),
           "pa_linear_int8_grouped")
    return outs

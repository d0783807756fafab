"""Pins of the oracle's weight-only INT8 linear layer against what the
definition fixes, computed independently of the oracle's loops: numpy fp64
matrix products of the dequantised weights, hand-built rounding cases and the
quantiser's round-trip bound ("PyTorch LLM Serving Engine", What is
implemented: symmetric per-output-channel INT8 weights)."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_240_gb300 import inputs as I


def _f64(bits, dtype):
    import dense_ref
    return dense_ref.bits_to_f64(bits, dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("m,n,k", [(1, 3, 5), (4, 16, 64), (7, 9, 130)])
def test_linear_equals_dense_product_of_dequantised_weights(dtype, m, n, k, olib):
    w = I.normal_bits((n, k), dtype, 1, m * n + k)
    x = I.normal_bits((m, k), dtype, 2, m * n + k)
    bias = I.normal_bits((n,), dtype, 3, m * n + k)
    codes, scales = oracle.quantize_weights(w, dtype, lib=olib)
    deq = codes.astype(np.float64) * scales.astype(np.float64)[:, None]
    ref = _f64(x, dtype) @ deq.T
    y = oracle.linear_int8(codes, scales, x, dtype, lib=olib)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    yb = oracle.linear_int8(codes, scales, x, dtype, bias_bits=bias, lib=olib)
    np.testing.assert_allclose(yb, ref + _f64(bias, dtype)[None, :], rtol=1e-12, atol=1e-12)


def test_weight_rows_follow_the_rounding_rule(olib):
    # row 0: amax 254 -> scale 2: 5/2 = 2.5 -> 2, -3/2 = -1.5 -> -2, 1/2 = 0.5 -> 0
    # row 1: amax 127 -> scale 1: 2.5 -> 2, 3.5 -> 4, -2.5 -> -2
    # row 2: all zero -> scale 0, codes 0
    rows = np.array([[254, 5, -3, 1], [127, 2.5, 3.5, -2.5], [0, 0, 0, 0]], np.float32)
    w = I.f32_to_bits(rows, "f16")
    codes, scales = oracle.quantize_weights(w, "f16", lib=olib)
    assert scales.tolist() == [2.0, 1.0, 0.0]
    assert codes.tolist() == [[127, 2, -2, 0], [127, 2, 4, -2], [0, 0, 0, 0]]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_quantised_weights_round_trip_within_half_a_step(dtype, olib):
    w = I.normal_bits((24, 96), dtype, 4, 0)
    codes, scales = oracle.quantize_weights(w, dtype, lib=olib)
    x = _f64(w, dtype)
    err = np.abs(x - codes.astype(np.float64) * scales.astype(np.float64)[:, None])
    assert (err <= scales.astype(np.float64)[:, None] / 2 * (1 + 2.0 ** -22)).all()
    top = np.argmax(np.abs(x), axis=1)
    assert (np.abs(codes[np.arange(24), top]) == 127).all()
    assert np.abs(codes).max() <= 127


def test_zero_activations_give_the_bias(olib):
    codes = np.ones((5, 8), np.int8)
    scales = np.full(5, 0.5, np.float32)
    x = np.zeros((2, 8), np.uint16)
    bias = I.f32_to_bits(np.array([1, -2, 0.25, 3, 0], np.float32), "bf16")
    y = oracle.linear_int8(codes, scales, x, "bf16", bias_bits=bias, lib=olib)
    assert y.tolist() == [[1, -2, 0.25, 3, 0]] * 2

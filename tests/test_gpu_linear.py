"""Weight-only INT8 linear on the GPU against the oracle ("PyTorch LLM Serving
Engine", What is implemented: symmetric per-output-channel INT8 weights, a
fused backend that reads the quantized tiles directly).

Quantisation is bit-exact (codes and scales).  Outputs are compared with the
fp64 oracle within the attention tolerance: activations ~N(0, 1) and weights
~N(0, 1/k) keep |y| near 1, where fp32 accumulation of k products (in a
different order) is far inside 2e-3 and the cast to fp16/bf16 inside 1e-2."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_240_gb300 as pa
from paged_kv_cache_240_gb300 import inputs as I
from paged_kv_cache_240_gb300 import linear as L
from gpu_util import TORCH_DT, assert_close, bits_to_torch

pytestmark = pytest.mark.gpu


def _weights(n, k, dtype, seed):
    w = np.random.default_rng([seed, 7]).standard_normal((n, k), dtype=np.float32)
    return I.f32_to_bits(w / np.sqrt(k), dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("n,k", [(16, 64), (48, 200), (7, 1000), (256, 4096)])
def test_quantize_bit_exact(dtype, n, k, olib):
    w = _weights(n, k, dtype, n + k)
    w[0, :] = 0                                   # an all-zero channel: scale 0
    codes_o, scales_o = oracle.quantize_weights(w, dtype, lib=olib)
    codes, scales = L.int8_quantize(bits_to_torch(w, dtype))
    torch.cuda.synchronize()
    assert (codes.cpu().numpy() == codes_o).all()
    assert (scales.cpu().numpy().view(np.uint32) == scales_o.view(np.uint32)).all()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("m,n,k", [(1, 16, 64), (3, 48, 192), (8, 64, 512), (13, 32, 256),
                                   (16, 128, 1024), (40, 16, 64), (5, 4096, 4096),
                                   (9, 80, 640), (2, 1008, 4672), (17, 336, 2048),
                                   (4, 16, 65536), (3, 5120, 640), (11, 9728, 576)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_linear_matches_oracle(dtype, m, n, k, with_bias, olib):
    """Ragged shapes (n = 80, 1008, 336 against 16-channel tiles; k = 640, 4672,
    576 against the 64-wide k blocks), token groups past 16, shapes whose
    thread blocks split k (small n: the workspace's partial sums and the
    reduce) and shapes that do not, and no workspace at all."""
    w = _weights(n, k, dtype, 3 * m + n + k)
    x = I.normal_bits((m, k), dtype, 11, m + n + k)
    bias = I.normal_bits((n,), dtype, 12, m + n + k) if with_bias else None
    codes, scales = L.int8_quantize(bits_to_torch(w, dtype))
    ref = oracle.linear_int8(codes.cpu().numpy(), scales.cpu().numpy(), x, dtype, bias_bits=bias,
                             lib=olib)
    xt = bits_to_torch(x, dtype)
    bt = bits_to_torch(bias, dtype) if with_bias else None
    nbytes = L.int8_workspace_bytes(m, n, k)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    for workspace in (ws, None):                  # split over k, and not
        y = L.int8_linear(codes, scales, xt, bias=bt, workspace=workspace)
        torch.cuda.synchronize()
        assert y.dtype == TORCH_DT[dtype] and y.shape == (m, n)
        assert_close(y.double().cpu().numpy(), ref,
                     "%s m=%d n=%d k=%d ws=%s" % (dtype, m, n, k, workspace is not None))


def test_linear_chain_shares_workspace(olib):
    """A chain of calls of different shapes back to back on one stream, all
    with one workspace (split and unsplit shapes mixed), repeated: every
    result matches the oracle and repeats give the same bits."""
    dtype = "bf16"
    shapes = [(8, 4096, 4096), (8, 1024, 11008), (3, 2048, 1024), (8, 5120, 640),
              (12, 9728, 576), (8, 4096, 4096)]
    # some of these calls split k (merged in the launch: no workspace needed)
    nbytes = max(L.int8_workspace_bytes(m, n, k) for m, n, k in shapes)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    mats = []
    for i, (m, n, k) in enumerate(shapes):
        w = _weights(n, k, dtype, 100 + i)
        x = I.normal_bits((m, k), dtype, 13, i)
        codes, scales = L.int8_quantize(bits_to_torch(w, dtype))
        mats.append((codes, scales, x, bits_to_torch(x, dtype)))
    outs = [[L.int8_linear(c, s, xt, workspace=ws) for c, s, _, xt in mats] for _ in range(3)]
    torch.cuda.synchronize()
    for j, (c, s, x, _) in enumerate(mats):
        ref = oracle.linear_int8(c.cpu().numpy(), s.cpu().numpy(), x, dtype, lib=olib)
        assert_close(outs[0][j].double().cpu().numpy(), ref, "chain %d" % j)
        for rep in (1, 2):
            assert torch.equal(outs[rep][j], outs[0][j])


def test_linear_rejects_bad_shapes_and_alignment():
    codes = torch.zeros((32, 128), dtype=torch.int8, device="cuda")
    scales = torch.ones(32, dtype=torch.float32, device="cuda")
    x = torch.zeros((2, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(pa.PaError) as e:          # n not a multiple of 16
        L.int8_linear(codes[:24], scales[:24], x)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    with pytest.raises(pa.PaError) as e:          # k not a multiple of 64
        L.int8_linear(codes[:, :96].contiguous(), scales, x[:, :96].contiguous())
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    xb = torch.zeros(2 * 128 + 1, dtype=torch.float16, device="cuda")[1:].view(2, 128)
    with pytest.raises(pa.PaError) as e:          # x not 16-byte aligned
        L.int8_linear(codes, scales, xb)
    assert e.value.status == pa.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("m,group,k", [
    (8, [4096, 4096, 4096], 4096),     # a 7B layer's q, k and v
    (8, [11008, 11008], 4096),         # gate and up
    (1, [16, 48, 1008, 336], 640),     # four ragged matrices, few channels: k split
    (13, [4096], 11008),               # one matrix, two token groups
    (3, [32, 16], 65536),              # very few channels over a long k: 8 splits
])
def test_grouped_linear_matches_oracle(dtype, m, group, k, olib):
    """One launch for the matrices that read the same activations; every
    output against the oracle, with a bias on every other matrix."""
    x = I.normal_bits((m, k), dtype, 21, m + k)
    xt = bits_to_torch(x, dtype)
    mats, refs = [], []
    for i, n in enumerate(group):
        w = _weights(n, k, dtype, 50 + i + k)
        bias = I.normal_bits((n,), dtype, 22, i) if i % 2 else None
        codes, scales = L.int8_quantize(bits_to_torch(w, dtype))
        mats.append((codes, scales, bits_to_torch(bias, dtype) if bias is not None else None))
        refs.append(oracle.linear_int8(codes.cpu().numpy(), scales.cpu().numpy(), x, dtype,
                                       bias_bits=bias, lib=olib))
    for rep in range(2):
        outs = L.int8_linear_grouped(mats, xt)
        torch.cuda.synchronize()
        for i, (y, ref) in enumerate(zip(outs, refs)):
            assert y.shape == (m, group[i]) and y.dtype == TORCH_DT[dtype]
            assert_close(y.double().cpu().numpy(), ref, "group %s matrix %d" % (group, i))
        if rep == 0:
            first = [y.clone() for y in outs]
        else:
            assert all(torch.equal(a, b) for a, b in zip(first, outs))  # same bits again

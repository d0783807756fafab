"""Parity at the benchmark's full sizes, in the launch configuration it times.

Each pool is built exactly as the benchmark builds it (bench.DeviceStep: seeded
device draws written through pa_write_kv in chunks of 32,768 history rows), one
step runs (the new tokens' write and the attention calls), and the outputs of
sampled sequences are recomputed by the oracle.  The oracle's inputs
are the generator's draws for those sequences' rows, drawn again chunk by chunk,
never what the kernels wrote: an int8 pool is quantised again by the oracle's own
writer.  The oracle keeps block i of a sequence in its physical block i, where
the device pool holds it wherever the shuffled block table says, so every check
is also one of invariance under block relabelling; the whole step is then run
again over a copy of the pool with its blocks permuted, and must give the same
bits.

A prefill chunk is checked on its first and last rows: the rows j0..j1-1 of a
chunk of C queries over a context of L keys see exactly what a chunk of j1-j0
queries over L-C+j1 keys sees (query j sees keys up to L-C+j and the window
behind it), so the oracle computes only those rows.

Collected after every other test, so that a run stopping at the first failure
has run the rest; each case builds a whole benchmark pool (up to ~3.5 GB).  The step runs as the
benchmark runs it (bench.DeviceStep.run): the write, then the attention calls;
with both decoding sequences and prefill chunks, the prefill on a second stream
launched before the decode."""
import pytest
import torch

import bench
import oracle
from full_size_util import (SEED, attend_relabelled, bits, check_sampled,
                            same_bits)
from paged_kv_cache_240_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["mha-7b", "int8-kv", "qwen2.5-1.5b", "mixed",
                                  "spec-verify"])
def test_full_size_step_sampled(name, olib):
    """The sampled outputs against the oracle, then the whole step's outputs
    again over a relabelled pool: bit for bit the same (no arithmetic depends
    on where a block lives)."""
    import paged_kv_cache_240_gb300 as pa
    from paged_kv_cache_240_gb300 import _build
    _build.build()
    w = I.make_workload(name, seed=SEED)
    st = bench.DeviceStep(w, torch, pa, I, SEED)
    st.run(torch.cuda.Stream())
    torch.cuda.synchronize()
    assert int(st.err[0]) == 0
    assert check_sampled(st, w, SEED, olib) > 0
    out_dec, out_pre, err = attend_relabelled(st, w, pa, SEED + 1)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    assert same_bits(out_dec, st.out_dec) and same_bits(out_pre, st.out_pre)


def test_full_size_int8_linear(olib):
    """The int8-linear workload's first layer exactly as the benchmark draws and
    runs it: grouped launches (q, k, v 4096x4096; o; gate, up 11008x4096; down
    4096x11008), 8 tokens; every output element against the oracle."""
    from gpu_util import assert_close
    from paged_kv_cache_240_gb300 import _build
    from paged_kv_cache_240_gb300 import linear as L
    _build.build()
    m = 8
    layer = bench.linear_layers(torch, bench.LINEAR_GROUPS, m, SEED)
    for x, mats in layer:
        L.int8_linear_grouped([(c, s, None) for c, s, _ in mats], x, outs=[y for _, _, y in mats])
    torch.cuda.synchronize()
    for x, mats in layer:
        for codes, scales, y in mats:
            n, k = codes.shape
            ref = oracle.linear_int8(codes.cpu().numpy(), scales.cpu().numpy(), bits(x), "bf16",
                                     lib=olib)
            assert_close(y.double().cpu().numpy(), ref,
                         "int8 linear %d tokens, n=%d k=%d" % (m, n, k))

"""pa_decode_noalloc against pa_decode, through the C ABI.

pa_decode_noalloc serves callers that are handed only their input and output
buffers and may not allocate device memory (a plugin inside an engine that owns
every allocation, or a serving loop that must not call cudaMalloc/cudaFree
because they can synchronise the device).  Its split-K partials live in scratch
compiled into the library instead of a caller-provided workspace.  This file is
collected after the other kernel tests (only the full-size sampled checks, which
build whole benchmark pools, come later) so that a run stopping at the first
failure has already run them; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_240_gb300 as pa
from paged_kv_cache_240_gb300 import _build
from paged_kv_cache_240_gb300 import inputs as I
from gpu_util import (ATOL, RTOL, assert_close, bits_to_torch, device_history, i32, new_err,
                      oracle_poison)

pytestmark = pytest.mark.gpu


# Batches with so few (sequence, kv head) units that the decode splits their
# contexts further than a thread-block cluster can merge: the split-K partials
# go through the scratch.
@pytest.mark.parametrize("name,kw", [
    ("qwen2.5-1.5b", dict(num_seqs=2, lens=("uniform", 1500, 4096))),
    ("int8-kv", dict(num_seqs=1, lens=("uniform", 3000, 8000))),
])
def test_noalloc_matches_pa_decode_twice(name, kw, olib):
    _build.build()
    w = I.make_workload(name, seed=17, **kw)
    kh, vh = I.history_rows(w)
    cache, err = device_history(w, kh, vh)
    cache_o = oracle.Cache(w.cache_dtype, w.num_blocks, w.num_kv_heads, w.head_dim)
    oracle_poison(cache_o, w.cache_dtype)
    oracle.write_kv(cache_o, kh, vh, I.source_dtype(w), w.history_slot_mapping(), lib=olib)
    B = w.num_decode
    need = pa.pa_decode_workspace_bytes(B, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                        w.max_blocks_per_seq, w.window)
    assert 0 < need <= pa.PA_NOALLOC_SCRATCH_BYTES  # the scratch really is used
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    tables, lens = i32(w.block_tables), i32(w.context_lens)
    sm = 1.0 / np.sqrt(w.head_dim)
    for call in range(2):  # the second call finds the first call's partials in the scratch
        q_bits = I.normal_bits((B, w.num_q_heads, w.head_dim), w.q_dtype, 40 + call, 7)
        q = bits_to_torch(q_bits, w.q_dtype)
        ref, got = torch.empty_like(q), torch.full_like(q, float("nan"))
        e1, e2 = new_err(), new_err()
        pa.pa_decode(cache, ref, q, tables, lens, sm, w.window, ws, e1)
        pa.pa_decode_noalloc(cache, got, q, tables, lens, sm, w.window, e2)
        torch.cuda.synchronize()
        assert int(e1[0]) == 0 and int(e2[0]) == 0
        r, g = ref.double().cpu().numpy(), got.double().cpu().numpy()
        assert np.isfinite(g).all()
        assert (np.abs(g - r) <= ATOL + RTOL * np.abs(r)).all(), (name, call)
        ref = oracle.attention(cache_o, q_bits, w.q_dtype, np.arange(B + 1, dtype=np.int32),
                               w.block_tables, w.context_lens, sm_scale=sm, window=w.window,
                               lib=olib)
        assert_close(g, ref, "%s call %d vs the oracle" % (name, call))


def test_noalloc_rejects_batches_beyond_its_scratch():
    _build.build()
    w = I.make_workload("int8-kv", seed=1, num_seqs=2, lens=("fixed", [16, 16]))
    cache, _ = device_history(w)
    B, MB = 1, 65536  # one sequence of up to 1M tokens: 1024 partitions of 64 blocks
    assert pa.pa_decode_workspace_bytes(B, 64, 8, 128, MB, 0) > pa.PA_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, 64, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    tables = torch.zeros((B, MB), dtype=torch.int32, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.pa_decode_noalloc(cache, out, q, tables, lens, 0.1, 0, new_err())
    assert e.value.status == pa.PA_ERR_UNSUPPORTED

"""pa_decode_append (one decode step in one launch: each sequence's new K/V row
written at its position L-1, then the attention) against pa_write_kv of those
slots followed by pa_decode, through the C ABI: the same output bits and the
same cache bytes, and the outputs within the tolerance of the oracle.  The
cases put the newest position at every offset of a block and in every warp's
share of a partition, over fp16, bf16 and int8 caches, with the workspace merge,
the in-launch cluster merge and a window."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_240_gb300 as pa
from paged_kv_cache_240_gb300 import inputs as I
from gpu_util import (assert_close, bits_to_torch, cache_bits, i32, new_err, oracle_poison,
                      poisoned_cache)

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny", dict(), None, None),
    ("qwen2.5-1.5b", dict(num_seqs=8, lens=("uniform", 1, 1400)), None, None),  # cluster merge
    ("qwen2.5-1.5b", dict(num_seqs=5, lens=("uniform", 1, 900)), 300, None),    # windowed
    ("int8-kv", dict(num_seqs=6, lens=("uniform", 1, 700)), None, None),        # int8, workspace
    ("mha-7b", dict(num_seqs=3, lens=("uniform", 17, 500)), None, None),
    # 16 query heads per kv head: two CTAs (row groups) hold each newest block and
    # both write the same bytes into it
    ("qwen2.5-1.5b", dict(num_seqs=4, lens=("uniform", 1, 900)), None, 16),
    ("int8-kv", dict(num_seqs=3, lens=("uniform", 1, 500)), None, 16),
]


def _history(w):
    """A poisoned device cache holding every position but each sequence's last,
    its flag word, and the step's new rows (K, V) and their slots."""
    kh, vh = I.history_rows(w)
    src = I.source_dtype(w)
    slots = w.history_slot_mapping()
    last = np.cumsum(w.context_lens) - 1  # each sequence's newest position
    prior = np.setdiff1d(np.arange(slots.size), last)
    cache = poisoned_cache(w)
    err = new_err()
    pa.pa_write_kv(cache, bits_to_torch(kh[prior], src), bits_to_torch(vh[prior], src),
                   i32(slots[prior]), err)
    return (cache, err, bits_to_torch(kh[last], src), bits_to_torch(vh[last], src),
            i32(slots[last]))


@pytest.mark.parametrize("name,kw,window,G", CASES)
def test_decode_append_matches_write_then_decode(name, kw, window, G, olib):
    w = I.make_workload(name, seed=77, window=window, **kw)
    if G is not None:
        w.num_kv_heads, w.num_q_heads = 2, 2 * G
    q_bits = I.query_rows(w)
    q = bits_to_torch(q_bits, w.q_dtype)
    tables, lens = i32(w.block_tables), i32(w.context_lens)
    sm = 1.0 / np.sqrt(w.head_dim)
    nbytes = pa.pa_decode_workspace_bytes(w.num_decode, w.num_q_heads, w.num_kv_heads,
                                          w.head_dim, w.max_blocks_per_seq, w.window)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    outs, caches = [], []
    for fused in (False, True):
        cache, err, k_new, v_new, slots = _history(w)
        out = torch.full_like(q, 7.0)
        if fused:
            pa.pa_decode_append(cache, k_new, v_new, out, q, tables, lens, sm, w.window, ws, err)
        else:
            pa.pa_write_kv(cache, k_new, v_new, slots, err)
            pa.pa_decode(cache, out, q, tables, lens, sm, w.window, ws, err)
        torch.cuda.synchronize()
        assert int(err[0]) == 0
        outs.append(out.view(torch.int16).cpu().numpy())
        caches.append(cache_bits(cache))
    assert np.array_equal(outs[0], outs[1])
    for a, b in zip(caches[0], caches[1]):
        assert np.array_equal(a, b)
    kh, vh = I.history_rows(w)
    oc = oracle.Cache(w.cache_dtype, w.num_blocks, w.num_kv_heads, w.head_dim)
    oracle_poison(oc, w.cache_dtype)
    oracle.write_kv(oc, kh, vh, I.source_dtype(w), w.history_slot_mapping(), lib=olib)
    ref = oracle.attention(oc, q_bits, w.q_dtype, w.cu_q_lens, w.block_tables, w.context_lens,
                           sm_scale=sm, window=w.window, lib=olib)
    got = torch.from_numpy(outs[1]).view(q.dtype).double().numpy()
    assert_close(got, ref, "pa_decode_append %s G=%s" % (name, G))


def test_decode_append_graph_replay_and_edge_rows():
    """Captured in a CUDA graph the launch replays to the same bits; a sequence
    of length 0 writes nothing and gets zeros; a sequence whose newest block id
    is outside the pool writes nothing and raises PA_FLAG_BLOCK_ID -- as
    pa_write_kv (which skips an out-of-range slot) + pa_decode do."""
    w = I.make_workload("qwen2.5-1.5b", seed=78, num_seqs=6, lens=("uniform", 20, 1200))
    q = bits_to_torch(I.query_rows(w), w.q_dtype)
    w.context_lens = w.context_lens.copy()
    tables_np = w.block_tables.copy()
    lens_np = w.context_lens.copy()
    lens_np[1] = 0
    tables_np[4, (lens_np[4] - 1) // 16] = w.num_blocks + 7
    tables, lens = i32(tables_np), i32(lens_np)
    sm = 1.0 / np.sqrt(w.head_dim)
    nbytes = pa.pa_decode_workspace_bytes(w.num_decode, w.num_q_heads, w.num_kv_heads,
                                          w.head_dim, w.max_blocks_per_seq, 0)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    res = []
    for mode in ("calls", "fused", "graph"):
        cache, err, k_new, v_new, slots = _history(w)
        # the calls' write skips what the fused launch skips: the empty sequence
        # and the one whose newest block is outside the pool
        slots_calls = slots.clone()
        slots_calls[1] = -1
        slots_calls[4] = w.num_blocks * 16 + 3  # out of range: skipped, PA_FLAG_SLOT_RANGE
        out = torch.full_like(q, 7.0)

        def call():
            if mode == "calls":
                pa.pa_write_kv(cache, k_new, v_new, slots_calls, err)
                pa.pa_decode(cache, out, q, tables, lens, sm, 0, ws, err)
            else:
                pa.pa_decode_append(cache, k_new, v_new, out, q, tables, lens, sm, 0, ws, err)

        stream = torch.cuda.Stream()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            if mode == "graph":
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    call()
                for _ in range(2):
                    out.fill_(7.0)
                    g.replay()
            else:
                call()
        torch.cuda.synchronize()
        flags = int(err[0])
        assert flags & pa.PA_FLAG_BLOCK_ID
        res.append((out.view(torch.int16).cpu().numpy(), cache_bits(cache)))
    for o, cb in res[1:]:
        assert np.array_equal(o, res[0][0])
        for a, b in zip(cb, res[0][1]):
            assert np.array_equal(a, b)
    out0 = torch.from_numpy(res[1][0]).view(q.dtype).float()
    assert (out0[1] == 0).all()

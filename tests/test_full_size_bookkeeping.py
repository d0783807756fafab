"""The full-size checks' bookkeeping, on the host (no GPU).

bench.DeviceStep is built on the host with a recording stand-in for pa_write_kv
that keeps the bits each slot received; the rows full_size_util draws again for
a sequence must be exactly the bits its slots hold, history and new tokens
alike, including sequences whose history straddles two chunks of the fill.  And
the reduction the full-size check makes for prefill chunks (rows j0..j1-1 of a
chunk of C queries over L keys computed as a chunk of j1-j0 queries over
L-C+j1 keys) gives the oracle's own rows, with and without a sliding window."""
import numpy as np
import pytest
import torch

import bench
import full_size_util as F
import oracle
from paged_kv_cache_240_gb300 import inputs as I


class RecordingPA:
    """Keeps, per slot, the K/V bits written there; computes nothing."""

    def __init__(self, w):
        n = w.num_blocks * w.block_size
        self.k = np.zeros((n, w.num_kv_heads, w.head_dim), np.uint16)
        self.v = np.zeros_like(self.k)
        self.written = np.zeros(n, np.int32)

    def PagedCache(self, *args):
        return None

    def pa_write_kv(self, cache, k, v, slots, err):
        s = slots.numpy()
        self.k[s] = F.bits(k)
        self.v[s] = F.bits(v)
        np.add.at(self.written, s, 1)

    def pa_decode_workspace_bytes(self, *args):
        return 0


def _checked_seqs(w):
    """First and last sequence and every one whose history straddles a chunk."""
    offs = F.history_offsets(w)
    pick = {0, w.num_seqs - 1}
    for b in range(w.num_seqs):
        if offs[b] // F.CHUNK != max(offs[b + 1] - 1, offs[b]) // F.CHUNK:
            pick.add(b)
    return sorted(pick)


@pytest.mark.parametrize("name,kw", [
    ("qwen2.5-1.5b", dict(num_seqs=24, lens=("uniform", 1000, 4000))),
    ("spec-verify", dict(num_chunks=40, chunk_len=9)),
])
def test_drawn_rows_are_the_written_rows(name, kw):
    seed = 5
    w = I.make_workload(name, seed=3, **kw)
    offs = F.history_offsets(w)
    assert offs[-1] > F.CHUNK                       # the fill takes several chunks
    rec = RecordingPA(w)
    st = bench.DeviceStep(w, torch, rec, I, seed, dev="cpu")
    st.write()
    cu = w.cu_q_lens
    assert (rec.written[w.history_slot_mapping()] == 1).all()
    seqs = _checked_seqs(w)
    assert len(seqs) > 2                            # some history straddles a chunk
    for b in seqs:
        L, C = int(w.context_lens[b]), int(w.q_lens[b])
        kh, vh = F.drawn_history(w, seed, int(offs[b]), int(offs[b + 1]), "cpu")
        s = w.slots(b, np.arange(L - C))
        assert np.array_equal(rec.k[s], kh) and np.array_equal(rec.v[s], vh), b
        s = w.slots(b, np.arange(L - C, L))
        assert np.array_equal(rec.k[s], F.bits(st.k_new[cu[b]:cu[b + 1]])), b
        assert np.array_equal(rec.v[s], F.bits(st.v_new[cu[b]:cu[b + 1]])), b


def test_empty_history_draws_nothing():
    w = I.make_workload("tiny", seed=1)
    kh, vh = F.drawn_history(w, 0, 7, 7, "cpu")
    assert kh.shape == (0, w.num_kv_heads, w.head_dim) == vh.shape


@pytest.mark.parametrize("window", [0, 20])
def test_chunk_rows_as_a_shorter_chunk(window, olib):
    w = I.make_workload("mixed", seed=4, num_seqs=1, lens=("fixed", [5]), num_chunks=1,
                        chunk_len=37, window=window)
    b = 1
    L, C = int(w.context_lens[b]), int(w.q_lens[b])
    src = I.source_dtype(w)
    k = I.normal_bits((L, w.num_kv_heads, w.head_dim), src, 9, 1)
    v = I.normal_bits((L, w.num_kv_heads, w.head_dim), src, 9, 2)
    q = I.normal_bits((C, w.num_q_heads, w.head_dim), w.q_dtype, 9, 3)
    nblk = -(-L // w.block_size)
    cache = oracle.Cache(w.cache_dtype, nblk, w.num_kv_heads, w.head_dim)
    oracle.write_kv(cache, k, v, src, np.arange(L, dtype=np.int32), lib=olib)
    table = np.arange(nblk, dtype=np.int32)[None, :]
    whole = oracle.attention(cache, q, w.q_dtype, np.array([0, C], np.int32), table,
                             np.array([L], np.int32), window=window, lib=olib)
    for j0, j1 in [(0, 9), (11, 12), (C - 9, C)]:
        part = oracle.attention(cache, q[j0:j1], w.q_dtype, np.array([0, j1 - j0], np.int32),
                                table, np.array([L - C + j1], np.int32), window=window,
                                lib=olib)
        assert np.array_equal(part, whole[j0:j1])

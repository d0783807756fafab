"""Speculative-decode verification on the GPU against the oracle.

A verification pass ("PyTorch LLM Serving Engine", What is implemented: one
target verification pass per proposal block; "llminfer", Speculative Decoding:
a target checking 8 assistant tokens) attends each sequence's last accepted
token and its drafts over the paged history, causally among themselves: the
chunked-prefill call with a few queries per sequence.  Rejected drafts are
rolled back by shortening the context ("MicroGen", Key Features: KV cache state
rollback on token rejection); their slots keep stale K/V that the next step
overwrites or never reads.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_240_gb300 as pa
from paged_kv_cache_240_gb300 import inputs as I
from gpu_util import (assert_close, bits_to_torch, device_history, i32, new_err, oracle_poison,
                      run_decode, run_prefill)

pytestmark = pytest.mark.gpu


def _verify_workload(seed, num_seqs, drafts, dtype="bf16", G=6, D=128, window=0):
    """spec-verify shapes shrunk to ``num_seqs`` sequences; sequence b verifies
    drafts[b] + 1 positions (ragged)."""
    w = I.make_workload("spec-verify", seed=seed, num_chunks=num_seqs, window=window)
    cache_dt, q_dt = (dtype.split("-") + [None])[:2]
    w.cache_dtype, w.q_dtype = cache_dt, q_dt or cache_dt
    w.num_kv_heads, w.num_q_heads, w.head_dim = 2, 2 * G, D
    C = np.asarray(drafts, np.int32) + 1
    w.q_lens = np.minimum(C, w.context_lens).astype(np.int32)
    return w


def _oracle_cache(olib, w):
    c = oracle.Cache(w.cache_dtype, w.num_blocks, w.num_kv_heads, w.head_dim)
    oracle_poison(c, w.cache_dtype)
    kh, vh = I.history_rows(w)
    oracle.write_kv(c, kh, vh, I.source_dtype(w), w.history_slot_mapping(), lib=olib)
    return c, kh, vh


def _verify(olib, w, sm):
    seqs = list(range(w.num_seqs))
    cache_o, kh, vh = _oracle_cache(olib, w)
    q = I.query_rows(w, seqs)
    ref = oracle.attention(cache_o, q, w.q_dtype, w.cu_q_lens, w.block_tables, w.context_lens,
                           sm_scale=sm, window=w.window, lib=olib)
    cache, err = device_history(w, kh, vh)
    got, flags = run_prefill(w, cache, q, sm, seqs)
    return got, ref, flags | int(err[0].item()), cache, cache_o


@pytest.mark.parametrize("dtype,G,D,window", [
    ("bf16", 6, 128, 0),      # the Qwen2.5-1.5B target's 12 q / 2 kv heads
    ("f16", 4, 128, 0),
    ("bf16", 6, 64, 300),
    ("i8-bf16", 4, 128, 0),   # verification over an int8 cache
    ("bf16", 1, 128, 0),
])
def test_verify_matches_oracle(dtype, G, D, window, olib):
    drafts = [8, 0, 3, 8, 5, 1, 7, 2]
    w = _verify_workload(7 + G + D, len(drafts), drafts, dtype, G, D, window)
    sm = 1.0 / np.sqrt(D)
    got, ref, flags, _, _ = _verify(olib, w, sm)
    assert flags == 0
    assert_close(got, ref, "verify %s G=%d D=%d W=%d" % (dtype, G, D, window))


@pytest.mark.parametrize("dtype,G,D,window,C", [
    ("bf16", 6, 128, 0, 9),     # 54 rows: both query slots on one tile's rows
    ("f16", 4, 64, 0, 32),      # 128 rows: the largest chunk that does so
    ("bf16", 4, 128, 0, 33),    # 132 rows: two query tiles, the second nearly empty
    ("bf16", 6, 128, 200, 9),   # a sliding window
])
def test_short_chunk_key_tiles(dtype, G, D, window, C, olib):
    """Chunks of a few queries over contexts chosen around the 128-key tiles:
    one key tile (the second query slot of a one-tile chunk gets none), two
    tiles, odd and even counts, and the context's partly written last block in
    either slot's tile (L = 9, 100, 128, 129, 200, 256, 257, 300, 383, 384, 520,
    1000, 1037)."""
    ctx = [9, 100, 128, 129, 200, 256, 257, 300, 383, 384, 520, 1000, 1037]
    w = I.make_workload("spec-verify", seed=90 + C + G, num_seqs=len(ctx), lens=("fixed", ctx),
                        num_chunks=0, window=window)
    cache_dt, q_dt = (dtype.split("-") + [None])[:2]
    w.cache_dtype, w.q_dtype = cache_dt, q_dt or cache_dt
    w.num_kv_heads, w.num_q_heads, w.head_dim = 2, 2 * G, D
    w.q_lens = np.minimum(C, w.context_lens).astype(np.int32)
    sm = 1.0 / np.sqrt(D)
    got, ref, flags, _, _ = _verify(olib, w, sm)
    assert flags == 0
    assert_close(got, ref, "short chunks %s G=%d D=%d W=%d C=%d" % (dtype, G, D, window, C))


@pytest.mark.parametrize("dtype", ["bf16", "i8-bf16"])
def test_rollback_then_decode(dtype, olib):
    """Verify 8 drafts, accept a random prefix of them, then decode the bonus
    token over the shortened context: the rejected drafts' stale slots must not
    be read (the first one is overwritten by the bonus token's K/V)."""
    drafts = [8, 8, 8, 8, 8, 8]
    w = _verify_workload(41, len(drafts), drafts, dtype, G=4, D=128)
    sm = 1.0 / np.sqrt(w.head_dim)
    got, ref, flags, cache, cache_o = _verify(olib, w, sm)
    assert flags == 0
    assert_close(got, ref, "verify before rollback")

    rng = np.random.default_rng(5)
    B = w.num_seqs
    # drafts kept per sequence (at most 7: the bonus token then lands in a slot
    # the block table already covers)
    accepted = rng.integers(0, 8, size=B)
    L, C = w.context_lens.astype(np.int64), w.q_lens.astype(np.int64)
    new_pos = L - C + 1 + accepted                   # where the bonus token goes
    assert (new_pos < L).all()
    slots = np.array([w.slots(b, [int(new_pos[b])])[0] for b in range(B)], np.int32)
    src = I.source_dtype(w)
    k_new = I.normal_bits((B, w.num_kv_heads, w.head_dim), src, w.seed, 777)
    v_new = I.normal_bits((B, w.num_kv_heads, w.head_dim), src, w.seed, 778)
    err = new_err()
    pa.pa_write_kv(cache, bits_to_torch(k_new, src), bits_to_torch(v_new, src), i32(slots), err)
    oracle.write_kv(cache_o, k_new, v_new, src, slots, lib=olib)

    dec = I.Workload(name="rollback", num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                     head_dim=w.head_dim, cache_dtype=w.cache_dtype, q_dtype=w.q_dtype,
                     window=w.window, num_blocks=w.num_blocks,
                     max_blocks_per_seq=w.max_blocks_per_seq,
                     context_lens=(new_pos + 1).astype(np.int32),
                     q_lens=np.ones(B, np.int32), block_tables=w.block_tables, seed=w.seed,
                     num_decode=B)
    q = I.normal_bits((B, w.num_q_heads, w.head_dim), w.q_dtype, w.seed, 779)
    ref_dec = oracle.attention(cache_o, q, w.q_dtype, dec.cu_q_lens, dec.block_tables,
                               dec.context_lens, sm_scale=sm, window=w.window, lib=olib)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    got_dec, dflags = run_decode(dec, cache, q, sm)
    assert dflags == 0
    assert_close(got_dec, ref_dec, "decode after rollback")

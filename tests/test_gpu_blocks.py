"""The block manager's tables and slots drive the kernels ("MicroGen", Key
Features: sliding window eviction): blocks evicted before the window are
poisoned (NaN), some are handed to another sequence, and a windowed decode and
a windowed chunk still match the oracle with no device flags."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_240_gb300 as pa
from paged_kv_cache_240_gb300 import inputs as I
from paged_kv_cache_240_gb300.blocks import BlockManager
from gpu_util import (POISON_AS_CODE, POISON_CODE, TORCH_DT, assert_close, bits_to_torch, i32, new_err,
                      oracle_poison)

pytestmark = pytest.mark.gpu

BS, NB, HKV, G, D, W = 16, 160, 2, 4, 128, 100


def _write(cache, cache_o, rows_k, rows_v, slots, src, olib):
    err = new_err()
    pa.pa_write_kv(cache, bits_to_torch(rows_k, src), bits_to_torch(rows_v, src), i32(slots), err)
    oracle.write_kv(cache_o, rows_k, rows_v, src, slots, lib=olib)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0


@pytest.mark.parametrize("dtype", ["bf16", "i8-bf16"])
def test_evicted_blocks_are_never_read(dtype, olib):
    cache_dt, q_dt = (dtype.split("-") + [None])[:2]
    q_dt = q_dt or cache_dt
    src = "bf16"
    lens = [300, 450, 81, 530]
    bm = BlockManager(NB, BS, max_seqs=5, max_blocks_per_seq=40, window=W)
    cache = pa.PagedCache(NB, HKV, D, cache_dt)
    cache_o = oracle.Cache(cache_dt, NB, HKV, D)
    oracle_poison(cache_o, cache_dt)
    if cache_dt == "i8":
        cache.k.fill_(POISON_CODE), cache.v.fill_(POISON_CODE)
        cache.k_scale.fill_(float("nan")), cache.v_scale.fill_(float("nan"))
    else:
        cache.k.fill_(float("nan")), cache.v.fill_(float("nan"))
    for s, L in enumerate(lens):  # prompts, then one decode token each
        for n in (L, 1):
            slots = bm.append(s, n)
            _write(cache, cache_o, I.normal_bits((n, HKV, D), src, 3, 10 * s + n),
                   I.normal_bits((n, HKV, D), src, 3, 10 * s + n + 5), slots, src, olib)
    freed = np.concatenate([bm.evict_window(s, L) for s, L in enumerate(lens)])
    assert freed.size > 0 and bm.stats()["evicted_blocks"] == freed.size
    # poison the evicted blocks on both sides, then give some of them to sequence 4
    for b in freed.tolist():
        if cache_dt == "i8":
            cache.k[b].fill_(POISON_CODE), cache.v[b].fill_(POISON_CODE)
            cache.k_scale[b].fill_(float("nan")), cache.v_scale[b].fill_(float("nan"))
        else:
            cache.k[b].fill_(float("nan")), cache.v[b].fill_(float("nan"))
    if cache_dt == "i8":
        cache_o.k[freed], cache_o.v[freed] = POISON_AS_CODE, POISON_AS_CODE
        cache_o.k_scale[freed], cache_o.v_scale[freed] = np.float32(np.nan), np.float32(np.nan)
    else:
        nan = torch.full((1,), float("nan"), dtype=TORCH_DT[cache_dt]).view(torch.int16).item()
        cache_o.k[freed], cache_o.v[freed] = np.uint16(nan & 0xFFFF), np.uint16(nan & 0xFFFF)
    s4 = bm.append(4, 70)
    _write(cache, cache_o, I.normal_bits((70, HKV, D), src, 3, 999),
           I.normal_bits((70, HKV, D), src, 3, 998), s4, src, olib)
    assert np.isin(s4 // BS, freed).any()  # the freed blocks are in use again

    seqs = np.arange(4, dtype=np.int32)
    tables, ctx = bm.tables(seqs)
    assert (tables == -1).any()
    sm = 1.0 / np.sqrt(D)
    Hq = HKV * G
    # windowed decode of each sequence's last token
    q = I.normal_bits((4, Hq, D), q_dt, 3, 4242)
    ref = oracle.attention(cache_o, q, q_dt, np.arange(5, dtype=np.int32), tables, ctx,
                           sm_scale=sm, window=W, lib=olib)
    out = torch.empty((4, Hq, D), dtype=TORCH_DT[q_dt], device="cuda")
    nbytes = pa.pa_decode_workspace_bytes(4, Hq, HKV, D, tables.shape[1], W)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    err = new_err()
    pa.pa_decode(cache, out, bits_to_torch(q, q_dt), i32(tables), i32(ctx), sm, W, ws, err)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    assert_close(out.double().cpu().numpy(), ref, "decode after eviction")
    # a windowed chunk of the last 7 positions of sequence 1: evict for its first query
    bm.evict_window(1, lens[1] + 1 - 7)
    tables, ctx = bm.tables(np.array([1], np.int32))
    qc = I.normal_bits((7, Hq, D), q_dt, 3, 4343)
    cu = np.array([0, 7], np.int32)
    refc = oracle.attention(cache_o, qc, q_dt, cu, tables, ctx, sm_scale=sm, window=W, lib=olib)
    outc = torch.empty((7, Hq, D), dtype=TORCH_DT[q_dt], device="cuda")
    err = new_err()
    pa.pa_prefill_chunk(cache, outc, bits_to_torch(qc, q_dt), i32(cu), 7, i32(tables), i32(ctx),
                        sm, W, err)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    assert_close(outc.double().cpu().numpy(), refc, "chunk after eviction")


@pytest.mark.parametrize("dtype", ["f16", "i8-bf16"])
def test_shared_prefix_blocks(dtype, olib):
    """Prefix caching: a prompt's full blocks are published; two later requests
    attach them (one all of them, one a prefix of them) and append their own
    tokens; decode and a chunk over the shared blocks match the oracle."""
    cache_dt, q_dt = (dtype.split("-") + [None])[:2]
    q_dt = q_dt or cache_dt
    src = "bf16" if cache_dt == "i8" else cache_dt
    bm = BlockManager(64, BS, max_seqs=3, max_blocks_per_seq=16)
    cache = pa.PagedCache(64, HKV, D, cache_dt)
    cache_o = oracle.Cache(cache_dt, 64, HKV, D)
    oracle_poison(cache_o, cache_dt)
    if cache_dt == "i8":
        cache.k.fill_(POISON_CODE), cache.v.fill_(POISON_CODE)
        cache.k_scale.fill_(float("nan")), cache.v_scale.fill_(float("nan"))
    else:
        cache.k.fill_(float("nan")), cache.v.fill_(float("nan"))

    def add(seq, n, stream):
        slots = bm.append(seq, n)
        _write(cache, cache_o, I.normal_bits((n, HKV, D), src, 5, stream),
               I.normal_bits((n, HKV, D), src, 5, stream + 1), slots, src, olib)

    add(0, 100, 10)                               # the shared prompt: 6 full blocks + 4
    keys = np.arange(1000, 1006, dtype=np.uint64)
    bm.publish(0, keys)
    assert bm.attach_prefix(1, keys) == 6         # the whole prompt prefix
    add(1, 30, 20)
    assert bm.attach_prefix(2, np.concatenate([keys[:3], [77]]).astype(np.uint64)) == 3
    add(2, 19, 30)
    assert bm.stats()["shared_blocks"] == 6
    for s in range(3):                            # one decode token each
        add(s, 1, 40 + 2 * s)
    tables, ctx = bm.tables(np.arange(3, dtype=np.int32))
    assert ctx.tolist() == [101, 127, 68]
    assert (tables[1, :6] == tables[0, :6]).all() and (tables[2, :3] == tables[0, :3]).all()
    sm = 1.0 / np.sqrt(D)
    Hq = HKV * G
    q = I.normal_bits((3, Hq, D), q_dt, 5, 4242)
    ref = oracle.attention(cache_o, q, q_dt, np.arange(4, dtype=np.int32), tables, ctx,
                           sm_scale=sm, window=0, lib=olib)
    out = torch.empty((3, Hq, D), dtype=TORCH_DT[q_dt], device="cuda")
    nbytes = pa.pa_decode_workspace_bytes(3, Hq, HKV, D, tables.shape[1], 0)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    err = new_err()
    pa.pa_decode(cache, out, bits_to_torch(q, q_dt), i32(tables), i32(ctx), sm, 0, ws, err)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    assert_close(out.double().cpu().numpy(), ref, "decode over shared blocks")
    # a chunk of the last 12 positions of sequence 1, over the shared prompt
    t1, c1 = bm.tables(np.array([1], np.int32))
    qc = I.normal_bits((12, Hq, D), q_dt, 5, 4343)
    cu = np.array([0, 12], np.int32)
    refc = oracle.attention(cache_o, qc, q_dt, cu, t1, c1, sm_scale=sm, window=0, lib=olib)
    outc = torch.empty((12, Hq, D), dtype=TORCH_DT[q_dt], device="cuda")
    err = new_err()
    pa.pa_prefill_chunk(cache, outc, bits_to_torch(qc, q_dt), i32(cu), 12, i32(t1), i32(c1), sm,
                        0, err)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    assert_close(outc.double().cpu().numpy(), refc, "chunk over shared blocks")


@pytest.mark.parametrize("dtype", ["bf16", "i8-bf16"])
def test_revived_prefix_blocks_after_the_request_ended(dtype, olib):
    """"llminfer", Prefix KV cache reuse: r1 writes and publishes its prompt,
    decodes and finishes; an unrelated request then needs more blocks than are
    free, so the cache gives back r1's last prompt block (least recently used);
    r2 with r1's prompt attaches the first five blocks from the cache, the other
    request rolls back three blocks, and r2 appends its own tokens.  Decode of
    both live requests matches the oracle."""
    cache_dt, q_dt = (dtype.split("-") + [None])[:2]
    q_dt = q_dt or cache_dt
    src = "bf16"
    nb = 18
    bm = BlockManager(nb, BS, max_seqs=3, max_blocks_per_seq=16)
    cache = pa.PagedCache(nb, HKV, D, cache_dt)
    cache_o = oracle.Cache(cache_dt, nb, HKV, D)
    oracle_poison(cache_o, cache_dt)
    if cache_dt == "i8":
        cache.k.fill_(POISON_CODE), cache.v.fill_(POISON_CODE)
        cache.k_scale.fill_(float("nan")), cache.v_scale.fill_(float("nan"))
    else:
        cache.k.fill_(float("nan")), cache.v.fill_(float("nan"))

    def add(seq, n, stream):
        slots = bm.append(seq, n)
        _write(cache, cache_o, I.normal_bits((n, HKV, D), src, 6, stream),
               I.normal_bits((n, HKV, D), src, 6, stream + 1), slots, src, olib)

    add(0, 100, 10)                               # r1's prompt: 6 full blocks + 4
    keys = np.arange(500, 506, dtype=np.uint64)
    bm.publish(0, keys)
    add(0, 1, 12)                                 # r1 decodes a token, then ends
    r1_table, _ = bm.tables(np.array([0], np.int32))
    bm.release(0)
    st = bm.stats()
    assert st["cached_blocks"] == 6 and st["free_blocks"] == nb - 6
    add(1, 16 * (nb - 6 + 1), 20)                 # all free blocks and one cached one
    assert bm.stats()["reclaimed_blocks"] == 1
    assert bm.attach_prefix(2, keys) == 5         # the prompt's last block was reclaimed
    bm.rollback(1, 48)                            # the other request gives back 3 blocks
    add(2, 20, 30)                                # r2 recomputes the rest of its prompt
    add(1, 1, 40)
    add(2, 1, 42)
    tables, ctx = bm.tables(np.array([1, 2], np.int32))
    assert (tables[1, :5] == r1_table[0, :5]).all()
    sm = 1.0 / np.sqrt(D)
    Hq = HKV * G
    q = I.normal_bits((2, Hq, D), q_dt, 6, 4444)
    ref = oracle.attention(cache_o, q, q_dt, np.arange(3, dtype=np.int32), tables, ctx,
                           sm_scale=sm, window=0, lib=olib)
    out = torch.empty((2, Hq, D), dtype=TORCH_DT[q_dt], device="cuda")
    nbytes = pa.pa_decode_workspace_bytes(2, Hq, HKV, D, tables.shape[1], 0)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    err = new_err()
    pa.pa_decode(cache, out, bits_to_torch(q, q_dt), i32(tables), i32(ctx), sm, 0, ws, err)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    assert_close(out.double().cpu().numpy(), ref, "decode over revived prefix blocks")

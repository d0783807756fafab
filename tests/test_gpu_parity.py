"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Write: int8 codes, scales and slot placement bit-exact (untouched slots keep
their poison).  Attention: |gpu - oracle| <= 2e-3 + 1e-2*|oracle| on every
output element, the flag word stays 0, and relabelling physical blocks gives a
bit-identical result.  Shapes are every workload's, shrunk so the oracle ends in
seconds, with ragged lengths spanning many blocks and partitions.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_checks as OC
import paged_kv_cache_240_gb300 as pa
from paged_kv_cache_240_gb300 import inputs as I
from gpu_util import (assert_close, bits_to_torch, cache_bits, codes_of_stored, device_history,
                      i32, new_err,
                      oracle_bits, oracle_poison, poisoned_cache, run_decode, run_prefill)

pytestmark = pytest.mark.gpu


def oracle_cache(olib, w):
    c = oracle.Cache(w.cache_dtype, w.num_blocks, w.num_kv_heads, w.head_dim)
    oracle_poison(c, w.cache_dtype)
    kh, vh = I.history_rows(w)
    oracle.write_kv(c, kh, vh, I.source_dtype(w), w.history_slot_mapping(), lib=olib)
    return c, kh, vh


def oracle_ref(olib, w, cache_o, seqs, sm):
    q = I.query_rows(w, seqs)
    cu = np.concatenate([[0], np.cumsum(w.q_lens[seqs])]).astype(np.int32)
    ref = oracle.attention(cache_o, q, w.q_dtype, cu, w.block_tables[seqs],
                           w.context_lens[seqs], sm_scale=sm, window=w.window, lib=olib)
    return q, ref


WRITE_CASES = [
    ("tiny", dict()),
    ("qwen2.5-1.5b", dict(num_seqs=3, lens=("uniform", 1, 200))),
    ("mha-7b", dict(num_seqs=2, lens=("uniform", 20, 90))),
    ("int8-kv", dict(num_seqs=4, lens=("uniform", 1, 300))),
    ("mixed", dict(num_seqs=3, num_chunks=2, chunk_len=37)),
]


@pytest.mark.parametrize("name,kw", WRITE_CASES, ids=[c[0] for c in WRITE_CASES])
def test_write_bit_exact(name, kw, olib):
    w = I.make_workload(name, seed=5, **kw)
    cache_o, kh, vh = oracle_cache(olib, w)
    cache, err = device_history(w, kh, vh)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    for g, o in zip(cache_bits(cache), oracle_bits(cache_o)):
        assert g.shape == o.shape and (g == o).all()


@pytest.mark.parametrize("src", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_write_int8_random_rows_and_padding(src, D, olib):
    rng = np.random.default_rng(D)
    NB, H, T = 13, 3, 150
    x = (rng.standard_normal((2, T, H, D)) * 10.0 ** rng.uniform(-4, 3, (2, T, H, 1)))
    x[0, 7] = 0.0  # all-zero rows: scale 0, codes 0
    kb, vb = I.f32_to_bits(x[0].astype(np.float32), src), I.f32_to_bits(x[1].astype(np.float32), src)
    slots = rng.choice(NB * 16, size=T, replace=False).astype(np.int32)
    slots[::11] = -1
    w = I.Workload("custom", H, H, D, "i8", src, 0, NB, 1, np.zeros(0, np.int32),
                   np.zeros(0, np.int32), np.zeros((0, 1), np.int32), 0, 0)
    cache = poisoned_cache(w)
    err = new_err()
    pa.pa_write_kv(cache, bits_to_torch(kb, src), bits_to_torch(vb, src), i32(slots), err)
    co = oracle.Cache("i8", NB, H, D)
    oracle_poison(co, "i8")
    assert oracle.write_kv(co, kb, vb, src, slots, lib=olib) == 0
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    for g, o in zip(cache_bits(cache), oracle_bits(co)):
        assert (g == o).all()


def test_write_golden_quant_cases():
    """The hand-derived tie cases, through the GPU quantiser."""
    for src in ("bf16", "f16"):
        for x, s, c in OC.read_quant_golden():
            D = 64
            row = np.zeros(D, np.float32)
            row[:8] = x
            w = I.Workload("custom", 1, 1, D, "i8", src, 0, 2, 1, np.zeros(0, np.int32),
                           np.zeros(0, np.int32), np.zeros((0, 1), np.int32), 0, 0)
            cache = poisoned_cache(w)
            bits = I.f32_to_bits(row, src).reshape(1, 1, D)
            err = new_err()
            pa.pa_write_kv(cache, bits_to_torch(bits, src), bits_to_torch(bits, src),
                           i32([17]), err)
            torch.cuda.synchronize()
            assert cache.k_scale[1, 0, 1].item() == s and cache.v_scale[1, 0, 1].item() == s
            # stored offset binary: byte = code + 128
            assert (codes_of_stored(cache.k[1, 0, 1, :8].cpu().numpy()).view(np.int8) == c).all()
            assert (codes_of_stored(cache.v[1, 0, 1, 8:].cpu().numpy()) == 0).all()


def test_write_out_of_range_slot_flagged():
    w = I.make_workload("tiny", seed=1)
    cache = poisoned_cache(w)
    before = cache_bits(cache)
    err = new_err()
    k = bits_to_torch(I.normal_bits((2, 2, 64), "f16", 0, 0), "f16")
    pa.pa_write_kv(cache, k, k, i32([w.num_blocks * 16, -1]), err)
    torch.cuda.synchronize()
    assert int(err[0]) == pa.PA_FLAG_SLOT_RANGE
    for a, b in zip(before, cache_bits(cache)):
        assert (a == b).all()


DECODE_CASES = [
    ("tiny", dict(), 0),
    ("tiny", dict(window=7), 0),
    ("qwen2.5-1.5b", dict(), 0),                                  # the full workload
    ("qwen2.5-1.5b", dict(num_seqs=4, window=300), 0),
    ("mha-7b", dict(num_seqs=3, lens=("uniform", 1, 700)), 0),
    ("mha-7b", dict(num_seqs=2, lens=("uniform", 600, 1500)), 3),  # forced small partitions
    ("mha-7b", dict(num_seqs=2, lens=("uniform", 600, 1500)), -5),  # 5-CTA clusters
    ("qwen2.5-1.5b", dict(num_seqs=3, window=700), -16),           # 16-CTA clusters
    ("int8-kv", dict(num_seqs=5, lens=("uniform", 1, 900)), 0),
    ("int8-kv", dict(num_seqs=3, lens=("uniform", 200, 700), window=100), 2),
    ("int8-kv", dict(num_seqs=3, lens=("uniform", 200, 700), window=100), -4),
    ("mixed", dict(num_seqs=6, num_chunks=1, chunk_len=20, lens=("uniform", 1, 2000)), 0),
]


@pytest.mark.parametrize("name,kw,pb", DECODE_CASES,
                         ids=["%s-%d" % (c[0], i) for i, c in enumerate(DECODE_CASES)])
def test_decode_matches_oracle(name, kw, pb, olib):
    w = I.make_workload(name, seed=11, **kw)
    sm = 1.0 / np.sqrt(w.head_dim)
    seqs = list(range(w.num_decode))
    cache_o, kh, vh = oracle_cache(olib, w)
    q, ref = oracle_ref(olib, w, cache_o, seqs, sm)
    cache, _ = device_history(w, kh, vh)
    got, flags = run_decode(w, cache, q, sm, partition_blocks=pb, seqs=seqs)
    assert flags == 0
    assert_close(got, ref, name)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "i8-f16", "i8-bf16"])
@pytest.mark.parametrize("G", [1, 3, 8, 16, 20])
def test_decode_shapes(D, dtype, G, olib):
    """Every cache type x head dim x GQA group (20 > 16 spans two row groups)."""
    cache_dt, q_dt = (dtype.split("-") + [None])[:2]
    q_dt = q_dt or cache_dt
    w = I.make_workload("qwen2.5-1.5b", seed=G + D, num_seqs=3, lens=("fixed", [1, 40, 77]))
    w.num_kv_heads, w.num_q_heads, w.head_dim = 2, 2 * G, D
    w.cache_dtype, w.q_dtype = cache_dt, q_dt
    sm = 0.7 / np.sqrt(D)
    cache_o, kh, vh = oracle_cache(olib, w)
    q, ref = oracle_ref(olib, w, cache_o, [0, 1, 2], sm)
    cache, _ = device_history(w, kh, vh)
    for pb in (0, 1, 2, -3, -16):  # workspace merges and cluster merges
        got, flags = run_decode(w, cache, q, sm, partition_blocks=pb)
        assert flags == 0
        assert_close(got, ref, "%s D=%d G=%d pb=%d" % (dtype, D, G, pb))


@pytest.mark.parametrize("pb", [4, -6])
def test_decode_block_relabelling_bit_identical(pb, olib):
    w = I.make_workload("int8-kv", seed=3, num_seqs=4, lens=("uniform", 50, 600))
    cache_o, kh, vh = oracle_cache(olib, w)
    q = I.query_rows(w)
    sm = 0.1
    cache, _ = device_history(w, kh, vh)
    a, fa = run_decode(w, cache, q, sm, partition_blocks=pb)
    perm = np.random.default_rng(1).permutation(w.num_blocks).astype(np.int32)
    w2 = I.make_workload("int8-kv", seed=3, num_seqs=4, lens=("uniform", 50, 600))
    w2.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1)
    cache2, _ = device_history(w2, kh, vh)
    b, fb = run_decode(w2, cache2, q, sm, partition_blocks=pb)
    assert fa == fb == 0
    assert (a == b).all()


@pytest.mark.parametrize("name,kw,pb", [
    ("qwen2.5-1.5b", dict(num_seqs=8, lens=("uniform", 1, 1500)), 8),
    ("int8-kv", dict(num_seqs=5, lens=("uniform", 100, 900)), 0),
    ("mha-7b", dict(num_seqs=3, lens=("uniform", 300, 700)), 1),
])
def test_decode_workspace_merge_scratch_and_reuse(name, kw, pb, olib):
    """The workspace merge (partition states in the caller's scratch, merged by
    a second kernel) needs no initialised workspace: scratch of all-ones bytes,
    random bytes or arbitrary 64-bit words, then the same workspace reused by
    repeated calls and by CUDA-graph replays, all give one result, bit for bit,
    within the tolerance of the oracle."""
    w = I.make_workload(name, seed=41, **kw)
    cache_o, kh, vh = oracle_cache(olib, w)
    cache, _ = device_history(w, kh, vh)
    seqs = list(range(w.num_decode))
    q_bits, ref = oracle_ref(olib, w, cache_o, seqs, 0.09)
    q = bits_to_torch(q_bits, w.q_dtype)
    tables, lens = i32(w.block_tables), i32(w.context_lens)
    nbytes = pa.pa_decode_workspace_bytes(w.num_decode, w.num_q_heads, w.num_kv_heads,
                                          w.head_dim, w.max_blocks_per_seq, w.window, pb)
    assert nbytes > 0  # the batch takes the workspace merge
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    err = new_err()
    out = torch.empty_like(q)

    def call():
        pa.pa_decode_partitioned(cache, out, q, tables, lens, 0.09, w.window, pb, ws, err)

    rng = np.random.default_rng(5)
    results = []
    fills = [lambda: ws.fill_(0xFF),
             lambda: ws.copy_(torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8))),
             # arbitrary 64-bit words
             lambda: ws.view(torch.int64)[: nbytes // 8].copy_(torch.from_numpy(
                 (rng.integers(1, 2 ** 39, nbytes // 8, dtype=np.int64) << 24)
                 | rng.integers(1, 8, nbytes // 8, dtype=np.int64)))]
    for fill in fills:
        fill()
        for _ in range(3):  # the same workspace, call after call
            out.fill_(7.0)
            call()
            torch.cuda.synchronize()
            results.append(out.double().cpu().numpy())
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
        for _ in range(3):  # replays repeat the captured launches
            out.fill_(7.0)
            g.replay()
            torch.cuda.synchronize()
            results.append(out.double().cpu().numpy())
    assert int(err[0]) == 0
    for r in results[1:]:
        assert (r == results[0]).all()
    assert_close(results[0], ref, "%s pb=%d" % (name, pb))


@pytest.mark.parametrize("pb", [0, -3])
def test_decode_empty_and_bad_data(pb, olib):
    """L = 0 gives zeros; a block id outside the pool drops its keys and sets
    PA_FLAG_BLOCK_ID; a context length above the table's reach is cut and sets
    PA_FLAG_CONTEXT_LEN -- both as the oracle's reading says."""
    w = I.make_workload("tiny", seed=8)
    cache_o, kh, vh = oracle_cache(olib, w)
    cache, _ = device_history(w, kh, vh)
    q = I.query_rows(w)
    w.context_lens = w.context_lens.copy()
    w.context_lens[0] = 0
    w.block_tables = w.block_tables.copy()
    w.block_tables[3, 1] = w.num_blocks + 100
    _, ref = oracle_ref(olib, w, cache_o, [0, 1, 2, 3], 0.125)
    got, flags = run_decode(w, cache, q, 0.125, partition_blocks=pb)
    assert flags == pa.PA_FLAG_BLOCK_ID
    assert (got[0] == 0).all()
    assert_close(got, ref, "bad block id")
    w.block_tables[3, 1] = w.block_tables[3, 0]  # restore a valid id
    w.context_lens[2] = 10 ** 6
    _, ref = oracle_ref(olib, w, cache_o, [0, 1, 2, 3], 0.125)
    got, flags = run_decode(w, cache, q, 0.125, partition_blocks=pb)
    assert flags & pa.PA_FLAG_CONTEXT_LEN
    assert_close(got[[0, 1, 3]], ref[[0, 1, 3]], "clamped length")


PREFILL_CASES = [
    ("mixed", dict(num_seqs=2, num_chunks=3, chunk_len=40, window=50)),
    ("mixed", dict(num_seqs=1, num_chunks=2, chunk_len=100, window=0)),
    ("mixed", dict(num_seqs=1, num_chunks=1, chunk_len=512)),        # full chunk, W = 2048
    ("int8-kv", dict(num_seqs=3, lens=("uniform", 30, 200))),        # decode as chunks of 1
]


@pytest.mark.parametrize("name,kw", PREFILL_CASES,
                         ids=["%s-%d" % (c[0], i) for i, c in enumerate(PREFILL_CASES)])
def test_prefill_matches_oracle(name, kw, olib):
    w = I.make_workload(name, seed=13, **kw)
    sm = 1.0 / np.sqrt(w.head_dim)
    seqs = list(range(w.num_seqs))
    cache_o, kh, vh = oracle_cache(olib, w)
    q, ref = oracle_ref(olib, w, cache_o, seqs, sm)
    cache, _ = device_history(w, kh, vh)
    got, flags = run_prefill(w, cache, q, sm, seqs)
    assert flags == 0
    assert_close(got, ref, name)


@pytest.mark.parametrize("dtype", ["f16", "i8-bf16"])
@pytest.mark.parametrize("G,D", [(1, 128), (3, 64), (8, 128)])
def test_prefill_shapes(dtype, G, D, olib):
    cache_dt, q_dt = (dtype.split("-") + [None])[:2]
    w = I.make_workload("mixed", seed=G * D, num_seqs=1, num_chunks=2, chunk_len=45, window=33)
    w.num_kv_heads, w.num_q_heads, w.head_dim = 2, 2 * G, D
    w.cache_dtype, w.q_dtype = cache_dt, q_dt or cache_dt
    sm = 0.5 / np.sqrt(D)
    seqs = [0, 1, 2]
    cache_o, kh, vh = oracle_cache(olib, w)
    q, ref = oracle_ref(olib, w, cache_o, seqs, sm)
    cache, _ = device_history(w, kh, vh)
    got, flags = run_prefill(w, cache, q, sm, seqs)
    assert flags == 0
    assert_close(got, ref, "%s G=%d D=%d" % (dtype, G, D))


def test_cuda_graph_replay_matches_direct_calls():
    """The calls only enqueue kernels on the caller's stream, so a CUDA graph of
    a step (write + decode + prefill) replays to the same bits as direct calls,
    also with the prefill on a second stream running beside the decode."""
    w = I.make_workload("mixed", seed=31, num_seqs=5, num_chunks=2, chunk_len=70, window=300)
    kh, vh = I.history_rows(w)
    nd = w.num_decode
    new = w.new_slot_mapping()
    hist_mask = ~np.isin(w.history_slot_mapping(), new)
    src = I.source_dtype(w)
    q = bits_to_torch(I.query_rows(w), w.q_dtype)
    nq = int(w.cu_q_lens[nd])
    q_dec, q_pre = q[:nq].clone(), q[nq:].clone()
    k_new = bits_to_torch(kh[~hist_mask], src)
    v_new = bits_to_torch(vh[~hist_mask], src)
    slots = i32(w.history_slot_mapping()[~hist_mask])
    tables_dec, tables_pre = i32(w.block_tables[:nd]), i32(w.block_tables[nd:])
    lens_dec, lens_pre = i32(w.context_lens[:nd]), i32(w.context_lens[nd:])
    cu = i32(w.cu_q_lens[nd:] - w.cu_q_lens[nd])
    sm = 1.0 / np.sqrt(w.head_dim)
    nbytes = pa.pa_decode_workspace_bytes(nd, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                          w.max_blocks_per_seq, w.window)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    outs = []
    for use_graph, two_streams in ((False, False), (True, False), (True, True)):
        cache = poisoned_cache(w)
        err = new_err()
        hs = w.history_slot_mapping()[hist_mask]
        pa.pa_write_kv(cache, bits_to_torch(kh[hist_mask], src), bits_to_torch(vh[hist_mask], src),
                       i32(hs), err)
        o_dec, o_pre = torch.empty_like(q_dec), torch.empty_like(q_pre)
        stream = torch.cuda.Stream()

        side = torch.cuda.Stream()

        def prefill():
            pa.pa_prefill_chunk(cache, o_pre, q_pre, cu, int(w.q_lens[nd:].max()), tables_pre,
                                lens_pre, sm, w.window, err)

        def step():
            pa.pa_write_kv(cache, k_new, v_new, slots, err)
            if two_streams:  # the prefill on a second stream, forked and joined in the graph
                cur = torch.cuda.current_stream()
                side.wait_stream(cur)
                with torch.cuda.stream(side):
                    prefill()
                pa.pa_decode(cache, o_dec, q_dec, tables_dec, lens_dec, sm, w.window, ws, err)
                cur.wait_stream(side)
            else:
                pa.pa_decode(cache, o_dec, q_dec, tables_dec, lens_dec, sm, w.window, ws, err)
                prefill()

        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            if use_graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    step()
                o_dec.zero_()
                o_pre.zero_()
                g.replay()
            else:
                step()
        torch.cuda.synchronize()
        assert int(err[0]) == 0
        outs.append((o_dec.clone(), o_pre.clone()))
    for o in outs[1:]:
        assert torch.equal(outs[0][0].view(torch.int16), o[0].view(torch.int16))
        assert torch.equal(outs[0][1].view(torch.int16), o[1].view(torch.int16))

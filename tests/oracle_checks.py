"""Pins of the CPU oracle against things other than itself.

Each ``check_*`` takes an oracle library handle and raises AssertionError when
the oracle disagrees with the pin.  ``test_oracle_pins.py`` runs them against the
oracle; ``test_oracle_mutants.py`` runs them against deliberately broken builds
of the oracle's source to show that every planted mistake trips at least one.

What pins what:
  * 16-bit decoding: exhaustive against numpy's binary16 and torch's bfloat16
    conversions, plus textbook values (tests/golden/float16_decode_cases.txt).
  * int8 quantiser: hand-derived tie cases (tests/golden/int8_quant_cases.txt),
    the round-to-nearest error bound, the code range and sign/monotonicity.
  * write: slot placement checked from the other direction (for each slot, which
    token names it); untouched slots keep their poison.
  * attention: torch SDPA in float64 on a contiguous cache (GQA by
    repeat_interleave, causal/window mask); brute force over every context
    length 1..64; closed forms (L=1, equal keys, q=0, W=1, W>=L); bit-identical
    results under a random relabelling of physical blocks; the online-softmax /
    split-K form against the two-pass definition.
  * INT8 linear: numpy's fp64 product of the dequantised weights (plus bias);
    weight rows quantised exactly as the KV cache write quantises a row.
"""
import os

import numpy as np
import torch

import oracle
from dense_ref import bits_to_f64, sdpa_dense
from paged_kv_cache_240_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ATOL = 1e-12


# ------------------------------------------------------------------ helpers

def build_cache(lib, w: I.Workload, poison=True):
    """Oracle cache holding every sequence's history, written by the oracle."""
    c = oracle.Cache(w.cache_dtype, w.num_blocks, w.num_kv_heads, w.head_dim)
    if poison:
        if w.cache_dtype == "i8":
            c.k_scale[:] = np.nan
            c.v_scale[:] = np.nan
        else:
            c.k[:] = I.NAN_BITS[w.cache_dtype]
            c.v[:] = I.NAN_BITS[w.cache_dtype]
    kh, vh = I.history_rows(w)
    bad = oracle.write_kv(c, kh, vh, I.source_dtype(w), w.history_slot_mapping(), lib=lib)
    assert bad == 0
    return c, kh, vh


def dense_rows(lib, w: I.Workload, rows_bits):
    """Values the cache holds for history rows, computed without the cache:
    16-bit rows decoded by numpy/torch; int8 rows quantised row by row with the
    oracle's quantiser (pinned on its own) and dequantised as code*scale."""
    src = I.source_dtype(w)
    x = bits_to_f64(rows_bits, src)
    if w.cache_dtype != "i8":
        return x
    out = np.empty_like(x)
    for idx in np.ndindex(x.shape[:-1]):
        codes, scale = oracle.quantize_row(x[idx].astype(np.float32), lib=lib)
        out[idx] = codes.astype(np.float64) * np.float64(scale)
    return out


def dense_reference(lib, w: I.Workload, kh, vh, q_bits, sm_scale):
    """SDPA over each sequence's contiguous history."""
    K, V = dense_rows(lib, w, kh), dense_rows(lib, w, vh)
    Q = bits_to_f64(q_bits, w.q_dtype)
    out = np.zeros(Q.shape)
    at_kv, cu = 0, w.cu_q_lens
    for b in range(w.num_seqs):
        L, C = int(w.context_lens[b]), int(w.q_lens[b])
        pos = np.arange(L - C, L)
        sl = slice(cu[b], cu[b + 1])
        out[sl] = sdpa_dense(Q[sl], K[at_kv:at_kv + L], V[at_kv:at_kv + L], pos,
                             w.window, sm_scale)
        at_kv += L
    return out


def oracle_attention(lib, w, cache, q_bits, sm_scale, online=None):
    args = (cache, q_bits, w.q_dtype, w.cu_q_lens, w.block_tables, w.context_lens)
    if online is None:
        return oracle.attention(*args, sm_scale=sm_scale, window=w.window, lib=lib)
    part, seg = online
    return oracle.attention_online(*args, sm_scale=sm_scale, window=w.window,
                                   part_tokens=part, seg_lens=seg, lib=lib)


def small_workloads():
    """Shapes of every workload, shrunk so fp64 SDPA finishes quickly, with
    ragged lengths and several blocks each."""
    return [
        I.make_workload("tiny", seed=3),
        I.make_workload("qwen2.5-1.5b", seed=1, num_seqs=3, lens=("uniform", 1, 90)),
        I.make_workload("mha-7b", seed=2, num_seqs=2, lens=("uniform", 20, 70)),
        I.make_workload("int8-kv", seed=4, num_seqs=3, lens=("uniform", 1, 80)),
        I.make_workload("mixed", seed=5, num_seqs=3, lens=("uniform", 1, 120), num_chunks=2,
                        chunk_len=9, window=40),
        I.make_workload("mixed", seed=6, num_seqs=2, lens=("uniform", 30, 60), num_chunks=1,
                        chunk_len=33, window=0),
    ]


# ------------------------------------------------------------------ 16-bit decoding

def check_f16_decode(lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([lib.pao_f16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    assert (np.signbit(got[~nan]) == np.signbit(ref[~nan])).all()


def check_bf16_decode(lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([lib.pao_bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def check_decode_golden(lib):
    with open(os.path.join(GOLDEN, "float16_decode_cases.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            dt, hx, val = line.split()
            fn = lib.pao_f16_to_double if dt == "f16" else lib.pao_bf16_to_double
            got = fn(int(hx, 16))
            assert got == float(val) and np.signbit(got) == np.signbit(float(val)), line


# ------------------------------------------------------------------ int8 quantiser

def read_quant_golden():
    cases = []
    with open(os.path.join(GOLDEN, "int8_quant_cases.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            xs, sc, cs = line.split("|")
            x = np.array([float(t) for t in xs.split(":")[1].split()], np.float32)
            s = np.float32(float(sc.split(":")[1]))
            c = np.array([int(t) for t in cs.split(":")[1].split()], np.int8)
            cases.append((x, s, c))
    return cases


def check_quant_golden(lib):
    for x, s, c in read_quant_golden():
        codes, scale = oracle.quantize_row(x, lib=lib)
        assert scale == s, (x, scale, s)
        assert (codes == c).all(), (x, codes, c)


def check_quant_golden_through_write(lib):
    """The same cases through the cache write, with bf16 and fp16 inputs."""
    for src in ("bf16", "f16"):
        for x, s, c in read_quant_golden():
            D = x.shape[0]
            cache = oracle.Cache("i8", 2, 1, D)
            bits = I.f32_to_bits(x, src).reshape(1, 1, D)
            oracle.write_kv(cache, bits, bits, src, np.array([17], np.int32), lib=lib)
            assert cache.k_scale[1, 0, 1] == s and cache.v_scale[1, 0, 1] == s
            assert (cache.k[1, 0, 1] == c).all() and (cache.v[1, 0, 1] == c).all()


def check_quant_properties(lib):
    rng = np.random.default_rng(7)
    for trial in range(300):
        D = [64, 128, 8, 3][trial % 4]
        mag = 10.0 ** rng.uniform(-6, 4)
        x = (rng.standard_normal(D) * mag).astype(np.float32)
        if trial % 5 == 0:
            x[rng.integers(D)] = 0
        codes, scale = oracle.quantize_row(x, lib=lib)
        amax = np.abs(x).max()
        assert abs(float(scale) - float(amax) / 127.0) <= float(amax) / 127.0 * 2.0 ** -23
        c = codes.astype(np.float64)
        assert np.abs(codes.astype(np.int32)).max() <= 127
        k = int(np.argmax(np.abs(x)))
        assert abs(int(codes[k])) == 127
        # nearest code: error at most half a step (plus the fp32 quotient rounding)
        err = np.abs(x.astype(np.float64) - c * float(scale))
        assert (err <= float(scale) * 0.5 * (1 + 2.0 ** -21)).all()
        assert (np.sign(c) * np.sign(x) >= 0).all()
        order = np.argsort(x, kind="stable")
        assert (np.diff(c[order]) >= 0).all()


# ------------------------------------------------------------------ write

def check_write_placement(lib):
    rng = np.random.default_rng(11)
    for dtype in ("f16", "bf16", "i8"):
        NB, H, D, S, T = 9, 3, 64, 16, 40
        cache = oracle.Cache(dtype, NB, H, D)
        if dtype == "i8":
            cache.k_scale[:] = -1.0
            cache.v_scale[:] = -2.0
        else:
            cache.k[:] = 0xABCD
            cache.v[:] = 0x1234
        slots = rng.choice(NB * S, size=T, replace=False).astype(np.int32)
        slots[::7] = -1                      # padding tokens
        slots[3] = NB * S + 5                # out of range: skipped and counted
        src = "bf16" if dtype == "i8" else dtype
        k = I.normal_bits((T, H, D), src, 1, 1)
        v = I.normal_bits((T, H, D), src, 1, 2)
        bad = oracle.write_kv(cache, k, v, src, slots, lib=lib)
        assert bad == 1
        for blk in range(NB):
            for off in range(S):
                who = np.nonzero(slots == blk * S + off)[0]
                for h in range(H):
                    if len(who) == 0:
                        if dtype == "i8":
                            assert cache.k_scale[blk, h, off] == -1.0
                            assert cache.v_scale[blk, h, off] == -2.0
                        else:
                            assert (cache.k[blk, h, off] == 0xABCD).all()
                            assert (cache.v[blk, h, off] == 0x1234).all()
                        continue
                    t = int(who[0])
                    if dtype == "i8":
                        for arr, sc, x in ((cache.k, cache.k_scale, k), (cache.v, cache.v_scale, v)):
                            codes, scale = oracle.quantize_row(
                                bits_to_f64(x[t, h], "bf16").astype(np.float32), lib=lib)
                            assert sc[blk, h, off] == scale
                            assert (arr[blk, h, off] == codes).all()
                    else:
                        assert (cache.k[blk, h, off] == k[t, h]).all()
                        assert (cache.v[blk, h, off] == v[t, h]).all()


# ------------------------------------------------------------------ attention

def check_dense_equivalence(lib):
    for w in small_workloads():
        cache, kh, vh = build_cache(lib, w)
        q = I.query_rows(w)
        sm = 1.0 / np.sqrt(w.head_dim)
        got = oracle_attention(lib, w, cache, q, sm)
        ref = dense_reference(lib, w, kh, vh, q, sm)
        assert np.isfinite(got).all()
        np.testing.assert_allclose(got, ref, rtol=0, atol=ATOL, err_msg=w.name)


def check_dense_windows(lib):
    """Windows smaller than, equal to and larger than the context, GQA 2 and 4."""
    for window in (1, 2, 5, 16, 17, 33, 64, 1000):
        for name, kw in (("tiny", {}), ("int8-kv", dict(num_seqs=2, lens=("uniform", 1, 50)))):
            w = I.make_workload(name, seed=window, window=window, **kw)
            cache, kh, vh = build_cache(lib, w)
            q = I.query_rows(w)
            got = oracle_attention(lib, w, cache, q, 0.3)
            ref = dense_reference(lib, w, kh, vh, q, 0.3)
            np.testing.assert_allclose(got, ref, rtol=0, atol=ATOL)


def check_brute_force_lengths(lib):
    """Every context length 1..64 on the tiny workload's shapes."""
    w = I.make_workload("tiny", seed=9, num_seqs=64, lens=("fixed", list(range(1, 65))))
    w.num_blocks = int((-(-w.context_lens // 16)).sum())
    perm = np.random.default_rng(5).permutation(w.num_blocks).astype(np.int32)
    w.block_tables[:] = -1
    at = 0
    for b in range(64):
        nb = -(-int(w.context_lens[b]) // 16)
        w.block_tables[b, :nb] = perm[at:at + nb]
        at += nb
    cache, kh, vh = build_cache(lib, w)
    q = I.query_rows(w)
    got = oracle_attention(lib, w, cache, q, 0.125)
    ref = dense_reference(lib, w, kh, vh, q, 0.125)
    np.testing.assert_allclose(got, ref, rtol=0, atol=ATOL)


def check_closed_forms(lib):
    w = I.make_workload("tiny", seed=21)
    cache, kh, vh = build_cache(lib, w)
    q = I.query_rows(w)
    V = bits_to_f64(vh, "f16")
    starts = np.concatenate([[0], np.cumsum(w.context_lens)])
    G = w.group
    # W = 1: each query sees only itself -> its own V row, exactly
    out = oracle.attention(cache, q, "f16", w.cu_q_lens, w.block_tables, w.context_lens,
                           window=1, lib=lib)
    for b in range(w.num_seqs):
        last = V[starts[b + 1] - 1]
        for h in range(w.num_q_heads):
            assert (out[b, h] == last[h // G]).all()
    # q = 0: uniform weights -> mean of the visible V rows
    zq = np.zeros_like(q)
    for window in (0, 7):
        out = oracle.attention(cache, zq, "f16", w.cu_q_lens, w.block_tables,
                               w.context_lens, window=window, lib=lib)
        for b in range(w.num_seqs):
            L = int(w.context_lens[b])
            lo = max(0, L - window) if window else 0
            mean = V[starts[b] + lo:starts[b] + L].mean(axis=0)
            for h in range(w.num_q_heads):
                np.testing.assert_allclose(out[b, h], mean[h // G], rtol=0, atol=ATOL)
    # W >= L is the same as no window, bit for bit
    a = oracle.attention(cache, q, "f16", w.cu_q_lens, w.block_tables, w.context_lens,
                         window=0, lib=lib)
    bb = oracle.attention(cache, q, "f16", w.cu_q_lens, w.block_tables, w.context_lens,
                          window=64, lib=lib)
    assert (a == bb).all()
    # L = 1: the only key's V row, exactly
    w1 = I.make_workload("tiny", seed=22, lens=("fixed", [1, 1, 1, 1]))
    c1, kh1, vh1 = build_cache(lib, w1)
    out = oracle.attention(c1, I.query_rows(w1), "f16", w1.cu_q_lens, w1.block_tables,
                           w1.context_lens, lib=lib)
    V1 = bits_to_f64(vh1, "f16")
    for b in range(4):
        for h in range(4):
            assert (out[b, h] == V1[b, h // 2]).all()
    # all keys equal -> mean of the V rows
    w2 = I.make_workload("tiny", seed=23)
    c2 = oracle.Cache("f16", w2.num_blocks, 2, 64)
    kh2, vh2 = I.history_rows(w2)
    kh2[:] = kh2[0]
    oracle.write_kv(c2, kh2, vh2, "f16", w2.history_slot_mapping(), lib=lib)
    out = oracle.attention(c2, I.query_rows(w2), "f16", w2.cu_q_lens, w2.block_tables,
                           w2.context_lens, lib=lib)
    V2 = bits_to_f64(vh2, "f16")
    for b in range(4):
        mean = V2[starts[b]:starts[b + 1]].mean(axis=0)
        for h in range(4):
            np.testing.assert_allclose(out[b, h], mean[h // 2], rtol=0, atol=ATOL)
    # empty context -> zeros
    w3 = I.make_workload("tiny", seed=24)
    w3.context_lens[:] = 0
    out = oracle.attention(cache, q, "f16", w3.cu_q_lens, w3.block_tables, w3.context_lens,
                           lib=lib)
    assert (out == 0).all()


def relabel_blocks(w: I.Workload, cache: oracle.Cache, seed: int):
    """Move every physical block to a new random place and rewrite the tables."""
    NB = w.num_blocks
    perm = np.random.default_rng(seed).permutation(NB).astype(np.int32)  # old -> new
    c2 = cache.copy()
    c2.k[perm] = cache.k
    c2.v[perm] = cache.v
    if cache.k_scale is not None:
        c2.k_scale[perm] = cache.k_scale
        c2.v_scale[perm] = cache.v_scale
    t2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1)
    return c2, t2.astype(np.int32)


def check_permutation_invariance(lib):
    for w in small_workloads():
        cache, _, _ = build_cache(lib, w)
        q = I.query_rows(w)
        a = oracle_attention(lib, w, cache, q, 0.1)
        c2, t2 = relabel_blocks(w, cache, 99)
        b = oracle.attention(c2, q, w.q_dtype, w.cu_q_lens, t2, w.context_lens,
                             sm_scale=0.1, window=w.window, lib=lib)
        assert (a == b).all(), w.name


def check_online_matches_two_pass(lib):
    rng = np.random.default_rng(31)
    for w in small_workloads():
        cache, _, _ = build_cache(lib, w)
        q = I.query_rows(w)
        a = oracle_attention(lib, w, cache, q, 0.2)
        for trial in range(3):
            part = int(rng.choice([1, 7, 16, 32, 48, 1000]))
            seg = rng.integers(1, 20, size=int(rng.integers(1, 5))).astype(np.int32)
            b = oracle_attention(lib, w, cache, q, 0.2, online=(part, seg))
            np.testing.assert_allclose(b, a, rtol=0, atol=ATOL)


def check_bad_block_ids_left_out(lib):
    """A block-table entry outside the pool drops that block's keys (reading for
    bad device data); the rest equals dense attention over the remaining keys."""
    w = I.make_workload("tiny", seed=41)
    cache, kh, vh = build_cache(lib, w)
    q = I.query_rows(w)
    w.block_tables[3, 1] = w.num_blocks + 3
    w.block_tables[2, 0] = -5
    got = oracle.attention(cache, q, "f16", w.cu_q_lens, w.block_tables, w.context_lens,
                           lib=lib)
    K, V, Q = bits_to_f64(kh, "f16"), bits_to_f64(vh, "f16"), bits_to_f64(q, "f16")
    starts = np.concatenate([[0], np.cumsum(w.context_lens)])
    for b in range(4):
        L = int(w.context_lens[b])
        keep = np.ones(L, bool)
        if b == 3:
            keep[16:32] = False
        if b == 2:
            keep[0:16] = False
        Kb, Vb = K[starts[b]:starts[b] + L][keep], V[starts[b]:starts[b] + L][keep]
        ref = sdpa_dense(Q[b:b + 1], Kb, Vb, [Kb.shape[0] - 1], 0, 1 / 8.0)
        np.testing.assert_allclose(got[b:b + 1], ref, rtol=0, atol=ATOL)


# ------------------------------------------------------------------ INT8 linear

def check_linear_dense(lib):
    """Weight-only INT8 linear = numpy's fp64 product of the dequantised weights
    (code * scale) with the activations, plus the bias; non-square shapes, both
    activation types."""
    for dtype in ("f16", "bf16"):
        for m, n, k in ((3, 5, 7), (2, 16, 64)):
            w = I.normal_bits((n, k), dtype, 21, m * n + k)
            x = I.normal_bits((m, k), dtype, 22, m * n + k)
            bias = I.normal_bits((n,), dtype, 23, m * n + k)
            codes, scales = oracle.quantize_weights(w, dtype, lib=lib)
            deq = codes.astype(np.float64) * scales.astype(np.float64)[:, None]
            ref = bits_to_f64(x, dtype) @ deq.T + bits_to_f64(bias, dtype)[None, :]
            y = oracle.linear_int8(codes, scales, x, dtype, bias_bits=bias, lib=lib)
            np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def check_linear_weight_rows_as_kv_rows(lib):
    """Each weight row (output channel) is quantised by the INT8 KV rule: the
    codes and scale equal what the cache write stores for the same row."""
    for dtype in ("f16", "bf16"):
        n, k = 6, 64
        w = I.normal_bits((n, k), dtype, 24, n)
        codes, scales = oracle.quantize_weights(w, dtype, lib=lib)
        cache = oracle.Cache("i8", 1, 1, k)
        rows = w.reshape(n, 1, k)
        oracle.write_kv(cache, rows, rows, dtype, np.arange(n, dtype=np.int32), lib=lib)
        assert (cache.k_scale[0, 0, :n] == scales).all(), (cache.k_scale[0, 0, :n], scales)
        assert (cache.k[0, 0, :n] == codes).all()


ALL_CHECKS = [  # cheap checks first: a mutant stops at the first failure
    check_linear_dense, check_linear_weight_rows_as_kv_rows,
    check_f16_decode, check_bf16_decode, check_decode_golden,
    check_quant_golden, check_quant_golden_through_write, check_quant_properties,
    check_write_placement,
    check_dense_equivalence, check_dense_windows, check_brute_force_lengths,
    check_closed_forms, check_permutation_invariance, check_online_matches_two_pass,
    check_bad_block_ids_left_out,
]

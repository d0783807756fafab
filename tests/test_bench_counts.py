"""The benchmark's algorithmic byte and flop counts (the numerators of its
roofline figures) against brute force on small workloads: every (query, key)
pair a query can see under the causal and window rules is enumerated, and the
K/V rows a call must read are the distinct keys any of its queries sees, once
per kv head; and the roofline object built from them."""
import numpy as np
import pytest

import bench
from paged_kv_cache_240_gb300 import inputs as I


def _visible(w, b):
    """(query position, key position) pairs of sequence b: a query at i sees j
    with i - W < j <= i (every j <= i without a window)."""
    L, C = int(w.context_lens[b]), int(w.q_lens[b])
    for i in range(L - C, L):
        for j in range(i + 1):
            if w.window == 0 or j > i - w.window:
                yield i, j


def _per_token_bytes(w):
    el = 1 if w.cache_dtype == "i8" else 2
    scales = 2 * 4 if w.cache_dtype == "i8" else 0  # one fp32 scale each for K and V
    return 2 * w.head_dim * el + scales


CASES = [
    ("mixed", dict(num_seqs=3, lens=("uniform", 1, 90), num_chunks=2, chunk_len=13, window=20)),
    ("mixed", dict(num_seqs=2, lens=("uniform", 1, 60), num_chunks=2, chunk_len=9, window=0)),
    ("int8-kv", dict(num_seqs=4, lens=("uniform", 1, 70))),
    ("spec-verify", dict(num_chunks=3, chunk_len=9, window=5)),
    ("qwen2.5-1.5b", dict(num_seqs=3, lens=("fixed", [1, 16, 33]))),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] + "-%d" % i for i, c in enumerate(CASES)])
def test_counts_match_brute_force(name, kw):
    w = I.make_workload(name, seed=7, **kw)
    per_tok = _per_token_bytes(w)
    dec_bytes = pre_bytes = flops = 0
    for b in range(w.num_seqs):
        pairs = list(_visible(w, b))
        keys = len({j for _, j in pairs})
        if b < w.num_decode:
            dec_bytes += keys * per_tok * w.num_kv_heads
        else:
            pre_bytes += keys * per_tok * w.num_kv_heads
            flops += len(pairs) * w.num_q_heads * 4 * w.head_dim
    assert bench.decode_kv_bytes(w) == dec_bytes
    assert bench.prefill_kv_bytes(w) == pre_bytes
    assert bench.prefill_flops(w) == flops
    assert w.kv_bytes() == dec_bytes + pre_bytes


def test_linear_bytes_by_definition():
    """Every code byte and fp32 scale once, each group's 16-bit activations in
    once (its matrices share them) and every output out."""
    m = 5
    groups = [[(48, 64), (32, 64)], [(16, 128)]]
    expect = 0
    for grp in groups:
        expect += m * grp[0][1] * 2                 # the group's activations
        for n, k in grp:
            expect += n * k * 1 + n * 4 + m * n * 2  # codes, scales, outputs
    assert bench.linear_bytes(m, groups) == expect


def test_recorded_traffic_only_for_unchanged_sources(tmp_path, monkeypatch):
    """The ncu traffic record is reported only while the hash of the kernel
    sources it names matches the sources as they are; otherwise null."""
    import json
    rec = {"kernel_sources": ["pa_decode.cu", "pa_device.cuh"],
           "traffic_bytes_per_launch": {"mha-7b": 123}}
    rec["kernel_source_hash"] = bench.kernel_source_hash(rec["kernel_sources"])
    good, stale = tmp_path / "good.json", tmp_path / "stale.json"
    good.write_text(json.dumps(rec))
    stale.write_text(json.dumps(dict(rec, kernel_source_hash="0" * 16)))
    monkeypatch.setitem(bench.TRAFFIC_FILES, "decode", str(good))
    assert bench.recorded_traffic("mha-7b") == 123
    assert bench.recorded_traffic("int8-kv") is None
    monkeypatch.setitem(bench.TRAFFIC_FILES, "decode", str(stale))
    assert bench.recorded_traffic("mha-7b") is None
    monkeypatch.setitem(bench.TRAFFIC_FILES, "decode", str(tmp_path / "missing.json"))
    assert bench.recorded_traffic("mha-7b") is None


PEAKS = {"hbm_gbs": 6792.1, "bf16_tflops": 1930.6, "bf16_tflops_sustained": 1716.1}


def test_roofline_picks_the_longer_call_and_its_bound():
    """mixed: the prefill call is longer and far above the machine balance
    (tensor); spec-verify: prefill longer, 54 flop per byte (HBM); mha-7b: the
    decode call (HBM).  achieved = algorithmic count / the call's time."""
    mixed = I.make_workload("mixed", seed=0)
    r = bench.roofline(mixed, 0.02, 0.08, PEAKS, "measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - bench.prefill_flops(mixed) / 0.08e-3 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 1930.6) < 1e-12
    assert abs(r["frac_of_nominal"] - r["achieved"] / 2250.0) < 1e-12
    sv = I.make_workload("spec-verify", seed=0)
    r = bench.roofline(sv, 0.0, 0.15, PEAKS, "measured")
    assert r["bound"] == "hbm" and "prefill" in r["kernel"]
    assert abs(r["achieved"] - bench.prefill_kv_bytes(sv) / 0.15e-3 / 1e9) < 1e-9
    mha = I.make_workload("mha-7b", seed=0)
    r = bench.roofline(mha, 0.37, 0.0, PEAKS, "measured")
    assert r["bound"] == "hbm" and "decode" in r["kernel"]
    assert abs(r["achieved"] - bench.decode_kv_bytes(mha) / 0.37e-3 / 1e9) < 1e-9
    assert abs(r["frac_of_nominal"] - r["achieved"] / 7900.0) < 1e-12


def test_roofline_traffic_only_for_full_size():
    w = I.make_workload("mha-7b", seed=0, num_seqs=16)
    r = bench.roofline(w, 0.1, 0.0, PEAKS, "measured", full_size=False)
    assert r["traffic"] is None and r["bound"] == "hbm"

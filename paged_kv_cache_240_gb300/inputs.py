"""Seeded synthetic workloads for the paged-KV attention path.

This module only draws random numbers and lays out the bookkeeping a serving
engine would hand to the kernels (context lengths, shuffled block tables, slot
mappings).  It holds none of the method's arithmetic: no quantisation, no
attention.  Both the CUDA path's tests/benchmark and the CPU oracle take their
inputs from here.

Workloads, shaped like the pages' (see the recipes in ``RECIPES``):
  * "PyTorch LLM Serving Engine", "Measured results": Qwen2.5-1.5B decode, batch
    8, a right-skewed (clipped log-normal) length mix.
  * same page, "What is implemented": fixed-size physical blocks, per-sequence
    block tables, chunked prefill sharing a step with decode.
  * "MicroGen", Key Features: dynamic INT8 KV quantisation, sliding window, GQA.
  * "llminfer", "Paged KV Cache And Continuous Batching": 16-token pages.
  * "llminfer", Speculative Decoding: a verification pass over 8 drafted tokens.

Every sequence's history (all positions before and including its new tokens) is
drawn as K/V rows ~N(0, 1).  A cache is built by writing that history through a
slot mapping, which each side does with its own write (the oracle's, or the
library's), so int8 codes are never produced here.  Physical blocks are a seeded
permutation of the pool, handed out to sequences in order; unused block-table
entries are -1.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BLOCK_SIZE = 16

# name -> recipe.  lens: ("fixed", [...]) | ("uniform", lo, hi) |
# ("lognormal", median, sigma, max)  (clipped to [1, max], rounded).
RECIPES = {
    "tiny": dict(num_seqs=4, lens=("fixed", [5, 17, 33, 64]), num_q_heads=4,
                 num_kv_heads=2, head_dim=64, cache_dtype="f16", q_dtype="f16",
                 max_context=64, num_blocks=32, window=0),
    "qwen2.5-1.5b": dict(num_seqs=8, lens=("lognormal", 512, 1.0, 4096), num_q_heads=12,
                         num_kv_heads=2, head_dim=128, cache_dtype="bf16",
                         q_dtype="bf16", max_context=4096, window=0),
    "mha-7b": dict(num_seqs=64, lens=("uniform", 1024, 4096), num_q_heads=32,
                   num_kv_heads=32, head_dim=128, cache_dtype="f16", q_dtype="f16",
                   max_context=4096, window=0),
    "int8-kv": dict(num_seqs=128, lens=("lognormal", 2048, 1.0, 8192), num_q_heads=32,
                    num_kv_heads=8, head_dim=128, cache_dtype="i8", q_dtype="bf16",
                    max_context=8192, window=0),
    # Speculative-decode verification ("llminfer", Speculative Decoding: a
    # Qwen2.5-1.5B target checking 8 assistant tokens; "PyTorch LLM Serving
    # Engine", What is implemented: one target verification pass per proposal
    # block): every sequence attends 9 new positions (the last accepted token and
    # 8 drafts) over its paged history, causally among themselves.  256 sequences,
    # prior context clipped log-normal around 2048.
    "spec-verify": dict(num_seqs=0, lens=("fixed", []), num_q_heads=12, num_kv_heads=2,
                        head_dim=128, cache_dtype="bf16", q_dtype="bf16", max_context=8192,
                        window=0, num_chunks=256, chunk_len=9,
                        prior=("lognormal", 2048, 1.0, 8192 - 9)),
    # 32 decode sequences plus 4 prefill chunks of 512 queries whose prior
    # context P0 ~ U[0, 3584] (so P0 + 512 <= 4096); sliding window 2048.
    "mixed": dict(num_seqs=32, lens=("uniform", 1, 4096), num_q_heads=32, num_kv_heads=8,
                  head_dim=128, cache_dtype="bf16", q_dtype="bf16", max_context=4096,
                  window=2048, num_chunks=4, chunk_len=512, prior=("uniform", 0, 3584)),
}


@dataclasses.dataclass
class Workload:
    """Bookkeeping of one step.  Sequences 0..num_decode-1 decode one token;
    the rest (mixed and spec-verify workloads) each attend a chunk of ``q_lens``
    new queries.
    ``context_lens`` count tokens after the step's write."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    cache_dtype: str
    q_dtype: str
    window: int
    num_blocks: int
    max_blocks_per_seq: int
    context_lens: np.ndarray   # int32 [B]
    q_lens: np.ndarray         # int32 [B]: new tokens (= queries) per sequence
    block_tables: np.ndarray   # int32 [B, MB], -1 where unused
    seed: int
    num_decode: int            # leading sequences that decode one token
    block_size: int = BLOCK_SIZE

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def cu_q_lens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def num_q_tokens(self) -> int:
        return int(self.q_lens.sum())

    def slots(self, seq: int, positions) -> np.ndarray:
        """Slot ids (physical_block*S + offset) of logical ``positions`` of ``seq``."""
        positions = np.asarray(positions, dtype=np.int64)
        blk = self.block_tables[seq, positions // self.block_size].astype(np.int64)
        return (blk * self.block_size + positions % self.block_size).astype(np.int32)

    def new_slot_mapping(self) -> np.ndarray:
        """Slots of the step's new tokens, in query-token order."""
        out = []
        for b in range(self.num_seqs):
            L, C = int(self.context_lens[b]), int(self.q_lens[b])
            out.append(self.slots(b, np.arange(L - C, L)))
        return np.concatenate(out).astype(np.int32) if out else np.zeros(0, np.int32)

    def history_slot_mapping(self, seqs=None) -> np.ndarray:
        """Slots of every position 0..L-1 of the given sequences, in order."""
        seqs = range(self.num_seqs) if seqs is None else seqs
        return np.concatenate([self.slots(b, np.arange(int(self.context_lens[b])))
                               for b in seqs] + [np.zeros(0, np.int32)]).astype(np.int32)

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one decode/prefill pass must read: every visible
        key's K and V row once per kv head (int8 adds the two fp32 scales)."""
        el = 1 if self.cache_dtype == "i8" else 2
        per_tok = 2 * self.head_dim * el + (8 if self.cache_dtype == "i8" else 0)
        total = 0
        for b in range(self.num_seqs):
            L, C = int(self.context_lens[b]), int(self.q_lens[b])
            lo_first = max(0, L - C - self.window + 1) if self.window > 0 else 0
            total += (L - lo_first) * per_tok * self.num_kv_heads
        return total


def _lengths(spec, n, rng):
    kind = spec[0]
    if kind == "fixed":
        return np.asarray(spec[1], np.int64)
    if kind == "uniform":
        return rng.integers(spec[1], spec[2] + 1, size=n)
    if kind == "lognormal":
        median, sigma, mx = spec[1], spec[2], spec[3]
        x = rng.lognormal(mean=math.log(median), sigma=sigma, size=n)
        return np.clip(np.rint(x), 1, mx).astype(np.int64)
    raise ValueError(spec)


def make_workload(name: str, seed: int = 0, num_seqs: int | None = None,
                  num_chunks: int | None = None, chunk_len: int | None = None,
                  window: int | None = None, lens=None) -> Workload:
    """Bookkeeping for workload ``name`` (overrides shrink it for parity runs)."""
    r = dict(RECIPES[name])
    rng = np.random.default_rng([seed, 1])
    B = num_seqs if num_seqs is not None else r["num_seqs"]
    L = _lengths(lens if lens is not None else r["lens"], B, rng)[:B]
    if L.shape[0] != B:
        raise ValueError("%s: %d decoding sequences but %d lengths given"
                         % (name, B, L.shape[0]))
    q_lens = np.ones(B, np.int64)
    if "num_chunks" in r:
        nc = num_chunks if num_chunks is not None else r["num_chunks"]
        C = chunk_len if chunk_len is not None else r["chunk_len"]
        prior = _lengths(r["prior"], nc, rng)
        prior = np.minimum(prior, r["max_context"] - C)
        L = np.concatenate([L, prior + C])
        q_lens = np.concatenate([q_lens, np.full(nc, C, np.int64)])
    S = BLOCK_SIZE
    MB = -(-r["max_context"] // S)
    need = -(-L // S)
    NB = r.get("num_blocks") or int(math.ceil(1.25 * need.sum()))
    NB = max(NB, int(need.sum()))
    perm = np.random.default_rng([seed, 2]).permutation(NB).astype(np.int32)
    tables = np.full((L.shape[0], MB), -1, np.int32)
    at = 0
    for b, nb in enumerate(need):
        tables[b, :nb] = perm[at:at + nb]
        at += nb
    return Workload(name=name, num_q_heads=r["num_q_heads"], num_kv_heads=r["num_kv_heads"],
                    head_dim=r["head_dim"], cache_dtype=r["cache_dtype"], q_dtype=r["q_dtype"],
                    window=r["window"] if window is None else window, num_blocks=NB,
                    max_blocks_per_seq=MB, context_lens=L.astype(np.int32),
                    q_lens=q_lens.astype(np.int32), block_tables=tables, seed=seed,
                    num_decode=B)


# --------------------------------------------------------------------------------
# random values (host, numpy): 16-bit bit patterns of N(0, 1) draws

def f32_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 draws -> fp16 or bf16 bit patterns (nearest-even rounding)."""
    x = np.ascontiguousarray(x, np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    raise ValueError(dtype)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """fp16 or bf16 bit patterns -> float32 (exact)."""
    bits = np.ascontiguousarray(bits, np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


def scaled_bits(bits: np.ndarray, dtype: str, factor) -> np.ndarray:
    """Draws of another magnitude: the values of ``bits`` times ``factor`` (a
    scalar, or an array broadcast against the rows, e.g. one factor per token),
    rounded back to ``dtype``."""
    x = bits_to_f32(bits, dtype).astype(np.float64) * np.asarray(factor, np.float64)
    return f32_to_bits(x.astype(np.float32), dtype)


def normal_bits(shape, dtype: str, seed: int, stream: int) -> np.ndarray:
    rng = np.random.default_rng([seed, 100 + stream])
    return f32_to_bits(rng.standard_normal(size=shape, dtype=np.float32), dtype)


def history_rows(w: Workload, seqs=None):
    """K and V rows (bits, [tokens, Hkv, D]) of every position of ``seqs`` in the
    order of :meth:`Workload.history_slot_mapping`.  Each sequence's rows come
    from its own stream, so a subset of sequences draws the same values."""
    seqs = range(w.num_seqs) if seqs is None else seqs
    src = "bf16" if w.cache_dtype == "i8" else w.cache_dtype
    ks, vs = [], []
    for b in seqs:
        L = int(w.context_lens[b])
        shape = (L, w.num_kv_heads, w.head_dim)
        ks.append(normal_bits(shape, src, w.seed, 2 * b + 1000))
        vs.append(normal_bits(shape, src, w.seed, 2 * b + 1001))
    z = np.zeros((0, w.num_kv_heads, w.head_dim), np.uint16)
    return np.concatenate(ks + [z]), np.concatenate(vs + [z])


def query_rows(w: Workload, seqs=None) -> np.ndarray:
    """q rows (bits, [tokens, Hq, D]) of the step's queries of ``seqs``."""
    seqs = range(w.num_seqs) if seqs is None else seqs
    qs = [normal_bits((int(w.q_lens[b]), w.num_q_heads, w.head_dim), w.q_dtype,
                      w.seed, 500000 + b) for b in seqs]
    return np.concatenate(qs + [np.zeros((0, w.num_q_heads, w.head_dim), np.uint16)])


def source_dtype(w: Workload) -> str:
    """dtype of the K/V rows the step writes (int8 caches quantise bf16 rows)."""
    return "bf16" if w.cache_dtype == "i8" else w.cache_dtype


NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}


# --------------------------------------------------------------------------------
# random values (device, torch): for pools too large to draw on the host quickly

def device_normal(shape, dtype: str, seed: int, stream: int, device="cuda"):
    """N(0, 1) draws made on ``device`` by torch's seeded generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + stream)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return t.to(torch.float16 if dtype == "f16" else torch.bfloat16)

"""Independent references used to pin the oracle (tests only).

Nothing here goes through block tables or the oracle's arithmetic: attention is
torch's own ``scaled_dot_product_attention`` in float64 on a contiguous
(position-ordered) cache, and 16-bit decoding is numpy's / torch's own.
"""
import numpy as np
import torch


def bits_to_f64(bits, dtype: str) -> np.ndarray:
    bits = np.ascontiguousarray(bits, np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
        return t.to(torch.float64).numpy()
    raise ValueError(dtype)


def visible_mask(positions, L: int, window: int) -> np.ndarray:
    """[C, L] bool: key j visible to a query at position i (j <= i, and
    j > i - window when window > 0)."""
    i = np.asarray(positions)[:, None]
    j = np.arange(L)[None, :]
    m = j <= i
    if window > 0:
        m &= j > i - window
    return m


def sdpa_dense(q, k, v, positions, window: int, sm_scale: float) -> np.ndarray:
    """q [C, Hq, D], k/v [L, Hkv, D] float64 (position order) -> [C, Hq, D].
    GQA: kv head g serves q heads g*G .. g*G+G-1 (repeat_interleave)."""
    C, Hq, D = q.shape
    L, Hkv, _ = k.shape
    out = np.zeros((C, Hq, D))
    if L == 0 or C == 0:
        return out
    G = Hq // Hkv
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    qt = torch.from_numpy(np.ascontiguousarray(q)).permute(1, 0, 2)[None]
    mask = visible_mask(positions, L, window)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(mask)[None, None], scale=sm_scale)
    o = o[0].permute(1, 0, 2).numpy().copy()
    o[~mask.any(axis=1)] = 0.0   # a query that sees no key returns zeros
    return o

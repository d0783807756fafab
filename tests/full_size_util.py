"""Bookkeeping of the full-size checks: which fill rows belong to a sequence,
the generator's draws for them made again, the oracle's recomputation of
sampled outputs, and the step rerun over a relabelled pool.  Plain host code
apart from the library calls of ``attend_relabelled``; the benchmark's pools
are built by bench.DeviceStep."""
import numpy as np
import torch

import bench
import oracle
from paged_kv_cache_240_gb300 import inputs as I

CHUNK = bench.FILL_CHUNK  # history rows per pa_write_kv of the benchmark's fill
SEED = 0            # the benchmark's default seed on rank 0
EDGE_ROWS = 48      # rows checked at each end of a prefill chunk


def bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def history_offsets(w):
    """Start of each sequence's history rows in the fill order: sequence by
    sequence, positions 0..L-C-1 of each."""
    n = (w.context_lens.astype(np.int64) - w.q_lens.astype(np.int64))
    return np.concatenate([[0], np.cumsum(n)])


def drawn_history(w, seed, lo, hi, dev):
    """K and V bits of fill rows lo..hi-1 as the generator drew them: each chunk
    of the fill is drawn again whole (its draws depend on its shape) and cut."""
    shape_tail = (w.num_kv_heads, w.head_dim)
    if hi <= lo:
        z = np.zeros((0,) + shape_tail, np.uint16)
        return z, z.copy()
    total = int(history_offsets(w)[-1])
    src = I.source_dtype(w)
    ks, vs = [], []
    for i in range((lo // CHUNK) * CHUNK, hi, CHUNK):
        n = min(CHUNK, total - i)
        a, z = max(lo, i) - i, min(hi, i + n) - i
        for out, stream in ((ks, 2 * i + 1), (vs, 2 * i + 2)):
            t = I.device_normal((n,) + shape_tail, src, seed, stream, dev)
            out.append(bits(t[a:z]))
    return np.concatenate(ks), np.concatenate(vs)


def sampled_seqs(w):
    """First, middle, last and longest of the decoding sequences and of the
    prefill chunks."""
    pick = set()
    for lo, hi in ((0, w.num_decode), (w.num_decode, w.num_seqs)):
        if hi > lo:
            pick |= {lo, (lo + hi - 1) // 2, hi - 1,
                     lo + int(np.argmax(w.context_lens[lo:hi]))}
    return sorted(pick)


def check_sampled(st, w, seed, olib, dev="cuda", seqs=None):
    """Compare the step's outputs of the sampled sequences with the oracle.
    Returns the number of output rows compared."""
    from gpu_util import assert_close
    cu = w.cu_q_lens
    nd = w.num_decode
    offs = history_offsets(w)
    src = I.source_dtype(w)
    k_new, v_new = bits(st.k_new), bits(st.v_new)
    rows = 0
    for b in (sampled_seqs(w) if seqs is None else seqs):
        L, C = int(w.context_lens[b]), int(w.q_lens[b])
        kh, vh = drawn_history(w, seed, int(offs[b]), int(offs[b + 1]), dev)
        assert kh.shape[0] == L - C
        k = np.concatenate([kh, k_new[cu[b]:cu[b + 1]]])
        v = np.concatenate([vh, v_new[cu[b]:cu[b + 1]]])
        nblk = -(-L // w.block_size)
        cache = oracle.Cache(w.cache_dtype, nblk, w.num_kv_heads, w.head_dim, w.block_size)
        assert oracle.write_kv(cache, k, v, src, np.arange(L, dtype=np.int32), lib=olib) == 0
        table = np.arange(nblk, dtype=np.int32)[None, :]
        if b < nd:
            q, out, base = st.q_dec, st.out_dec, 0
        else:
            q, out, base = st.q_pre, st.out_pre, int(cu[nd])
        q_rows = bits(q[cu[b] - base:cu[b + 1] - base])
        got_rows = out[cu[b] - base:cu[b + 1] - base].double().cpu().numpy()
        spans = [(0, C)] if C <= 2 * EDGE_ROWS else [(0, EDGE_ROWS), (C - EDGE_ROWS, C)]
        for j0, j1 in spans:
            ref = oracle.attention(cache, q_rows[j0:j1], w.q_dtype,
                                   np.array([0, j1 - j0], np.int32), table,
                                   np.array([L - C + j1], np.int32), sm_scale=st.sm,
                                   window=w.window, lib=olib)
            assert_close(got_rows[j0:j1], ref,
                         "%s: sequence %d (context %d, %d new), rows %d..%d"
                         % (w.name, b, L, C, j0, j1 - 1))
            rows += j1 - j0
    return rows


def attend_relabelled(st, w, pa, seed):
    """The step's attention again, over a copy of the pool whose physical blocks
    are permuted (block b moves to perm[b]; the tables are mapped alike).
    Returns (out_dec, out_pre, flags)."""
    c = st.cache
    perm = torch.from_numpy(np.random.default_rng(seed).permutation(w.num_blocks)).to(c.k.device)
    c2 = pa.PagedCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.cache_dtype)
    for name in ("k", "v", "k_scale", "v_scale"):
        if getattr(c, name) is not None:
            getattr(c2, name)[perm] = getattr(c, name)

    def mapped(t):
        return torch.where(t >= 0, perm[t.clamp(min=0).long()].to(torch.int32), t).contiguous()

    out_dec, out_pre = torch.empty_like(st.out_dec), torch.empty_like(st.out_pre)
    err = torch.zeros_like(st.err)
    if st.nd:
        pa.pa_decode(c2, out_dec, st.q_dec, mapped(st.tables_dec), st.lens_dec, st.sm,
                     w.window, st.ws, err)
    if st.max_q:
        pa.pa_prefill_chunk(c2, out_pre, st.q_pre, st.cu, st.max_q, mapped(st.tables_pre),
                            st.lens_pre, st.sm, w.window, err)
    return out_dec, out_pre, err


def same_bits(a, b):
    return a.shape == b.shape and torch.equal(a.view(torch.int16), b.view(torch.int16))

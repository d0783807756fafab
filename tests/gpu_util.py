"""Helpers for the GPU tests: put a workload on the device through the library's
own write, and compare against the oracle within the stated tolerance."""
import numpy as np
import torch

import paged_kv_cache_240_gb300 as pa
from paged_kv_cache_240_gb300 import inputs as I

# fp16/bf16 attention outputs vs the fp64 oracle: |gpu - ref| <= ATOL + RTOL*|ref|
ATOL, RTOL = 2e-3, 1e-2

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}
POISON_CODE = 0x55  # int8 cache bytes of slots nothing wrote (stored form)
# An int8 cache stores each code c as the offset-binary byte c + 128 (include/pa.h);
# the oracle keeps the codes themselves.  POISON_CODE as a stored byte stands for
# this code:
POISON_AS_CODE = int(np.uint8(POISON_CODE ^ 0x80).view(np.int8))  # as the oracle's int8


def codes_of_stored(stored):
    """Offset-binary cache bytes (numpy uint8/int8) -> the codes' bytes (uint8)."""
    return stored.view(np.uint8) ^ np.uint8(0x80)


def bits_to_torch(bits: np.ndarray, dtype: str, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy())
    return t.view(TORCH_DT[dtype]).to(device)


def i32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def new_err():
    return torch.zeros(4, dtype=torch.int32, device="cuda")


def poisoned_cache(w: I.Workload) -> pa.PagedCache:
    """Device cache whose every slot starts as poison: NaN for 16-bit caches,
    NaN scales and POISON_CODE codes for int8."""
    c = pa.PagedCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.cache_dtype)
    if w.cache_dtype == "i8":
        c.k.fill_(POISON_CODE)
        c.v.fill_(POISON_CODE)
        c.k_scale.fill_(float("nan"))
        c.v_scale.fill_(float("nan"))
    else:
        c.k.fill_(float("nan"))
        c.v.fill_(float("nan"))
    return c


def oracle_poison(cache_o, dtype):
    """The same poison on the oracle's host cache, bit for bit."""
    if dtype == "i8":
        cache_o.k[:] = POISON_AS_CODE
        cache_o.v[:] = POISON_AS_CODE
        cache_o.k_scale[:] = np.float32(np.nan)
        cache_o.v_scale[:] = np.float32(np.nan)
    else:
        nan = torch.full((1,), float("nan"), dtype=TORCH_DT[dtype]).view(torch.int16).item()
        cache_o.k[:] = np.uint16(nan & 0xFFFF)
        cache_o.v[:] = np.uint16(nan & 0xFFFF)


def device_history(w: I.Workload, kh=None, vh=None):
    """Poisoned device cache holding every sequence's history, written by
    pa_write_kv.  Returns (cache, err_flag)."""
    if kh is None:
        kh, vh = I.history_rows(w)
    src = I.source_dtype(w)
    cache = poisoned_cache(w)
    err = new_err()
    slots = w.history_slot_mapping()
    if slots.size:
        pa.pa_write_kv(cache, bits_to_torch(kh, src), bits_to_torch(vh, src), i32(slots), err)
    return cache, err


def cache_bits(cache: pa.PagedCache):
    """Bytes of a device cache (K, V and scales) on the host, in the oracle's
    form: an int8 cache's offset-binary bytes become the codes' bytes."""
    out = [cache.k.view(torch.int8).cpu().numpy().view(np.uint8),
           cache.v.view(torch.int8).cpu().numpy().view(np.uint8)]
    if cache.k_scale is not None:
        out = [codes_of_stored(b) for b in out]
        out += [cache.k_scale.cpu().numpy().view(np.uint32),
                cache.v_scale.cpu().numpy().view(np.uint32)]
    return out


def oracle_bits(cache_o):
    out = [cache_o.k.view(np.uint8), cache_o.v.view(np.uint8)]
    if cache_o.k_scale is not None:
        out += [cache_o.k_scale.view(np.uint32), cache_o.v_scale.view(np.uint32)]
    return out


def run_decode(w: I.Workload, cache, q_bits, sm_scale, partition_blocks=0, seqs=None):
    """pa_decode over the decode sequences of ``w``.  Returns (out fp64, flags)."""
    seqs = list(range(w.num_decode)) if seqs is None else seqs
    q = bits_to_torch(q_bits, w.q_dtype)
    B = len(seqs)
    out = torch.empty_like(q)
    tables = i32(w.block_tables[seqs])
    lens = i32(w.context_lens[seqs])
    nbytes = pa.pa_decode_workspace_bytes(B, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                          w.max_blocks_per_seq, w.window, partition_blocks)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    err = new_err()
    pa.pa_decode_partitioned(cache, out, q, tables, lens, sm_scale, w.window, partition_blocks,
                             ws, err)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), int(err[0].item())


def run_prefill(w: I.Workload, cache, q_bits, sm_scale, seqs):
    """pa_prefill_chunk over sequences ``seqs`` of ``w``.  Returns (out, flags)."""
    q = bits_to_torch(q_bits, w.q_dtype)
    qlens = w.q_lens[seqs]
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    out = torch.empty_like(q)
    err = new_err()
    pa.pa_prefill_chunk(cache, out, q, i32(cu), int(qlens.max()), i32(w.block_tables[seqs]),
                        i32(w.context_lens[seqs]), sm_scale, w.window, err)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), int(err[0].item())


def assert_close(got, ref, what=""):
    assert got.shape == ref.shape
    bad = ~(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.abs(got - ref)[bad].max()
        raise AssertionError("%s: %d of %d elements outside tolerance (worst |diff| %.3g); "
                             "first at %s: got %s ref %s" % (
                                 what, bad.sum(), bad.size, worst, idx.tolist(),
                                 got[tuple(idx[0])], ref[tuple(idx[0])]))

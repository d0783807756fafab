"""ctypes binding of include/pa_blocks.h: the host-side manager of the paged KV
cache's physical blocks (argument marshalling only; the logic is the C++ library's)."""
from __future__ import annotations

import ctypes

import numpy as np

from . import PaError, load_library, PA_OK


class _Stats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int), ("free_blocks", ctypes.c_int),
                ("live_seqs", ctypes.c_int), ("tokens_held", ctypes.c_longlong),
                ("preemptions", ctypes.c_longlong), ("recompute_tokens", ctypes.c_longlong),
                ("evicted_blocks", ctypes.c_longlong), ("rolled_back_tokens", ctypes.c_longlong),
                ("published_blocks", ctypes.c_longlong), ("prefix_hit_blocks", ctypes.c_longlong),
                ("shared_blocks", ctypes.c_int), ("cached_blocks", ctypes.c_int),
                ("revived_blocks", ctypes.c_longlong), ("reclaimed_blocks", ctypes.c_longlong)]


def _lib():
    lib = load_library()
    if not getattr(lib, "_pa_blocks_ready", False):
        P, I = ctypes.c_void_p, ctypes.c_int
        i32p = ctypes.POINTER(ctypes.c_int32)
        lib.pa_blocks_create.argtypes = [I, I, I, I, I]
        lib.pa_blocks_create.restype = P
        lib.pa_blocks_destroy.argtypes = [P]
        lib.pa_blocks_destroy.restype = None
        lib.pa_blocks_append.argtypes = [P, I, I, i32p]
        lib.pa_blocks_rollback.argtypes = [P, I, I]
        lib.pa_blocks_release.argtypes = [P, I]
        lib.pa_blocks_preempt.argtypes = [P, I]
        lib.pa_blocks_evict_window.argtypes = [P, I, I, i32p, I]
        lib.pa_blocks_tables.argtypes = [P, i32p, I, i32p, i32p]
        lib.pa_blocks_context_len.argtypes = [P, I]
        lib.pa_blocks_get_stats.argtypes = [P, ctypes.POINTER(_Stats)]
        u64p = ctypes.POINTER(ctypes.c_uint64)
        lib.pa_blocks_publish.argtypes = [P, I, u64p, I]
        lib.pa_blocks_attach_prefix.argtypes = [P, I, u64p, I]
        for name in ("pa_blocks_append", "pa_blocks_rollback", "pa_blocks_release",
                     "pa_blocks_preempt", "pa_blocks_evict_window", "pa_blocks_tables",
                     "pa_blocks_context_len", "pa_blocks_get_stats", "pa_blocks_publish",
                     "pa_blocks_attach_prefix"):
            getattr(lib, name).restype = I
        lib._pa_blocks_ready = True
    return lib


def _i32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if a is not None else None


def _check(status, what):
    if status != PA_OK:
        raise PaError(status, what)


class BlockManager:
    """A pool of ``num_blocks`` blocks of ``block_size`` tokens for sequences
    0..max_seqs-1 (see include/pa_blocks.h)."""

    def __init__(self, num_blocks, block_size=16, max_seqs=1, max_blocks_per_seq=1, window=0):
        self._lib = _lib()
        self.block_size, self.max_seqs = block_size, max_seqs
        self.max_blocks_per_seq = max_blocks_per_seq
        self._h = self._lib.pa_blocks_create(num_blocks, block_size, max_seqs,
                                             max_blocks_per_seq, window)
        if not self._h:
            raise ValueError("pa_blocks_create rejected the sizes")

    def close(self):
        if self._h:
            self._lib.pa_blocks_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def append(self, seq: int, num_tokens: int) -> np.ndarray:
        """Slots of the new positions (int32)."""
        out = np.empty(max(num_tokens, 0), np.int32)
        _check(self._lib.pa_blocks_append(self._h, seq, num_tokens, _i32p(out)),
               "pa_blocks_append")
        return out

    def rollback(self, seq: int, num_tokens: int):
        _check(self._lib.pa_blocks_rollback(self._h, seq, num_tokens), "pa_blocks_rollback")

    def release(self, seq: int):
        _check(self._lib.pa_blocks_release(self._h, seq), "pa_blocks_release")

    def preempt(self, seq: int):
        _check(self._lib.pa_blocks_preempt(self._h, seq), "pa_blocks_preempt")

    def evict_window(self, seq: int, oldest_query: int) -> np.ndarray:
        """Ids of the blocks freed (as many as the sequence has)."""
        cap = self.max_blocks_per_seq
        out = np.empty(cap, np.int32)
        n = self._lib.pa_blocks_evict_window(self._h, seq, oldest_query, _i32p(out), cap)
        if n < 0:
            raise PaError(1, "pa_blocks_evict_window")
        return out[:n].copy()

    def tables(self, seqs):
        """(block_tables [n, max_blocks_per_seq], context_lens [n]) as int32."""
        seqs = np.ascontiguousarray(seqs, np.int32)
        tab = np.empty((seqs.size, self.max_blocks_per_seq), np.int32)
        lens = np.empty(seqs.size, np.int32)
        _check(self._lib.pa_blocks_tables(self._h, _i32p(seqs), seqs.size, _i32p(tab),
                                          _i32p(lens)), "pa_blocks_tables")
        return tab, lens

    def publish(self, seq: int, keys):
        """Register seq's first len(keys) (full) blocks under the given prefix keys."""
        keys = np.ascontiguousarray(keys, np.uint64)
        _check(self._lib.pa_blocks_publish(
            self._h, seq, keys.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), keys.size),
            "pa_blocks_publish")

    def attach_prefix(self, seq: int, keys) -> int:
        """Attach the longest run of registered blocks matching keys to the empty
        sequence seq; returns how many blocks were attached."""
        keys = np.ascontiguousarray(keys, np.uint64)
        k = self._lib.pa_blocks_attach_prefix(
            self._h, seq, keys.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), keys.size)
        if k < 0:
            raise PaError(1, "pa_blocks_attach_prefix")
        return k

    def context_len(self, seq: int) -> int:
        n = self._lib.pa_blocks_context_len(self._h, seq)
        if n < 0:
            raise PaError(1, "pa_blocks_context_len")
        return n

    def stats(self) -> dict:
        st = _Stats()
        _check(self._lib.pa_blocks_get_stats(self._h, ctypes.byref(st)), "pa_blocks_get_stats")
        return {f: getattr(st, f) for f, _ in _Stats._fields_}

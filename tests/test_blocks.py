"""Host-side block manager (include/pa_blocks.h): no GPU.

The C++ library is checked against the contract its header states, and against
a plain Python model of that contract over random operation sequences
("PyTorch LLM Serving Engine", What is implemented: fixed-size blocks, block
tables, an O(1) free-list allocator, memory accounting, recomputation counters
after preemption; "MicroGen", Key Features: sliding window eviction, rollback).
"""
import numpy as np
import pytest

import paged_kv_cache_240_gb300 as pa
from paged_kv_cache_240_gb300 import _build
from paged_kv_cache_240_gb300.blocks import BlockManager


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def check_invariants(bm, nseq, shared_ok=False):
    tab, lens = bm.tables(np.arange(nseq))
    owned = tab[tab >= 0]
    st = bm.stats()
    distinct = len(set(owned.tolist()))
    if not shared_ok:
        assert distinct == owned.size, "a block in two places"
    assert st["shared_blocks"] == owned.size - distinct or shared_ok
    assert distinct + st["free_blocks"] + st["cached_blocks"] == st["num_blocks"]
    assert st["tokens_held"] == int(lens.sum())
    assert st["live_seqs"] == int((lens > 0).sum())
    for s in range(nseq):
        need = -(-int(lens[s]) // bm.block_size)
        assert (tab[s, need:] == -1).all(), "blocks past the context"
    return tab, lens


def test_append_slots_follow_the_table():
    bm = BlockManager(num_blocks=10, block_size=16, max_seqs=3, max_blocks_per_seq=4)
    s0 = bm.append(0, 20)           # two blocks
    s1 = bm.append(1, 5)            # one block
    s0b = bm.append(0, 13)          # fills block 1, takes block 2... (33 tokens -> 3 blocks)
    tab, lens = check_invariants(bm, 3)
    assert lens.tolist() == [33, 5, 0]
    for seq, slots, first in ((0, s0, 0), (1, s1, 0), (0, s0b, 20)):
        pos = np.arange(first, first + slots.size)
        assert (slots == tab[seq, pos // 16] * 16 + pos % 16).all()
    assert bm.stats()["free_blocks"] == 10 - 4


def test_append_is_all_or_nothing():
    bm = BlockManager(num_blocks=3, block_size=16, max_seqs=2, max_blocks_per_seq=8)
    bm.append(0, 40)                # 3 blocks: the pool is empty
    before = bm.tables([0, 1])
    with pytest.raises(pa.PaError) as e:
        bm.append(1, 1)
    assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
    with pytest.raises(pa.PaError) as e:
        bm.append(0, 9)             # 49 tokens need a 4th block
    assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
    bm.append(0, 8)                 # 48 still fits the last block
    after = bm.tables([0, 1])
    assert (after[0] == before[0]).all() and after[1].tolist() == [48, 0]
    small = BlockManager(num_blocks=100, block_size=16, max_seqs=1, max_blocks_per_seq=2)
    with pytest.raises(pa.PaError) as e:
        small.append(0, 33)         # more than max_blocks_per_seq blocks
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    assert small.context_len(0) == 0


def test_free_list_reuses_freed_blocks_first():
    bm = BlockManager(num_blocks=8, block_size=4, max_seqs=4, max_blocks_per_seq=8)
    bm.append(0, 8)                 # blocks 0, 1
    bm.append(1, 4)                 # block 2
    tab, _ = bm.tables([0])
    bm.release(0)
    got = bm.append(2, 4)           # takes the most recently freed block
    assert got[0] // 4 in tab[0].tolist()
    check_invariants(bm, 4)


def test_rollback_frees_emptied_blocks():
    bm = BlockManager(num_blocks=6, block_size=16, max_seqs=2, max_blocks_per_seq=6)
    bm.append(0, 30)
    bm.append(0, 9)                 # 39 tokens, 3 blocks (speculative drafts)
    bm.rollback(0, 8)               # 31: the third block empties
    tab, lens = check_invariants(bm, 2)
    assert lens[0] == 31 and tab[0, 2] == -1
    st = bm.stats()
    assert st["rolled_back_tokens"] == 8 and st["free_blocks"] == 4
    again = bm.append(0, 1)         # position 31 reuses the second block's last slot
    assert again[0] == tab[0, 1] * 16 + 15
    with pytest.raises(pa.PaError):
        bm.rollback(0, 33)
    bm.rollback(0, 32)
    check_invariants(bm, 2)
    assert bm.stats()["live_seqs"] == 0


def test_preemption_counts_recomputation():
    bm = BlockManager(num_blocks=8, block_size=16, max_seqs=3, max_blocks_per_seq=8)
    bm.append(0, 50)
    bm.append(1, 10)
    bm.preempt(0)
    bm.preempt(2)                   # empty: nothing to count
    st = bm.stats()
    assert st["preemptions"] == 1 and st["recompute_tokens"] == 50
    assert bm.context_len(0) == 0 and st["free_blocks"] == 8 - 1
    check_invariants(bm, 3)


def test_window_eviction_frees_only_blocks_no_query_can_see():
    W = 40
    bm = BlockManager(num_blocks=20, block_size=16, max_seqs=2, max_blocks_per_seq=20, window=W)
    bm.append(0, 150)               # blocks 0..9
    tab0, _ = bm.tables([0])
    # next query at position 150 sees keys 111..150: blocks 0..5 (positions < 96) go
    freed = bm.evict_window(0, 150)
    assert sorted(freed.tolist()) == sorted(tab0[0, :6].tolist())
    tab, lens = check_invariants(bm, 2)
    assert (tab[0, :6] == -1).all() and (tab[0, 6:10] >= 0).all() and lens[0] == 150
    assert bm.evict_window(0, 150).size == 0          # idempotent
    assert bm.stats()["evicted_blocks"] == 6
    # the window's first key (111) sits in block 6: it stays
    assert tab[0, 6] == tab0[0, 6]
    # a rollback must leave the next query's window (keys L2-39 .. L2) in kept blocks
    with pytest.raises(pa.PaError):
        bm.rollback(0, 150 - 134)                     # query 134 would need key 95
    bm.rollback(0, 150 - 135)                         # query 135 needs keys 96.. : fine
    assert bm.context_len(0) == 135
    nowin = BlockManager(num_blocks=4, block_size=16, max_seqs=1, max_blocks_per_seq=4)
    nowin.append(0, 60)
    assert nowin.evict_window(0, 1000).size == 0      # no window: nothing to evict


def test_bad_arguments():
    bm = BlockManager(num_blocks=4, block_size=16, max_seqs=2, max_blocks_per_seq=4)
    for call in (lambda: bm.append(2, 1), lambda: bm.append(-1, 1), lambda: bm.append(0, -1),
                 lambda: bm.rollback(0, 1), lambda: bm.release(5), lambda: bm.preempt(-2),
                 lambda: bm.tables([3]), lambda: bm.context_len(7),
                 lambda: bm.evict_window(9, 0)):
        with pytest.raises(pa.PaError):
            call()
    with pytest.raises(ValueError):
        BlockManager(num_blocks=0)
    assert bm.append(0, 0).size == 0


class Model:
    """The header's contract in plain Python."""

    def __init__(self, nb, bs, ns, mb, w):
        self.bs, self.mb, self.w = bs, mb, w
        self.free = list(range(nb - 1, -1, -1))
        self.tab = [[-1] * mb for _ in range(ns)]
        self.lens = [0] * ns
        self.kept = [0] * ns

    def nblk(self, n):
        return -(-n // self.bs)

    def append(self, s, n):
        have, need = self.nblk(self.lens[s]), self.nblk(self.lens[s] + n)
        if need > self.mb:
            return "unsupported"
        if need - have > len(self.free):
            return "out"
        for i in range(have, need):
            self.tab[s][i] = self.free.pop()
        self.lens[s] += n
        return "ok"

    def rollback(self, s, n):
        L2 = self.lens[s] - n
        if n < 0 or L2 < 0 or (self.kept[s] > 0 and L2 - self.w + 1 < self.kept[s] * self.bs):
            return "bad"
        for i in range(self.nblk(L2), self.nblk(self.lens[s])):
            self.free.append(self.tab[s][i])
            self.tab[s][i] = -1
        self.lens[s] = L2
        return "ok"

    def drop(self, s):
        for i in range(self.kept[s], self.nblk(self.lens[s])):
            if self.tab[s][i] >= 0:
                self.free.append(self.tab[s][i])
                self.tab[s][i] = -1
        self.lens[s], self.kept[s] = 0, 0

    def evict(self, s, oldest):
        if self.w <= 0 or oldest - self.w + 1 <= 0:
            return []
        upto = min((oldest - self.w + 1) // self.bs, self.nblk(self.lens[s]))
        out = []
        for i in range(self.kept[s], upto):
            if self.tab[s][i] >= 0:
                out.append(self.tab[s][i])
                self.free.append(self.tab[s][i])
                self.tab[s][i] = -1
        self.kept[s] = max(self.kept[s], upto)
        return out


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_model(seed):
    rng = np.random.default_rng(seed)
    nb, bs, ns, mb, w = 40, int(rng.choice([4, 16])), 5, 12, int(rng.choice([0, 23, 64]))
    bm = BlockManager(nb, bs, ns, mb, w)
    m = Model(nb, bs, ns, mb, w)
    for _ in range(400):
        s = int(rng.integers(ns))
        op = rng.choice(["append", "append", "rollback", "release", "preempt", "evict"])
        if op == "append":
            n = int(rng.integers(0, 30))
            want = m.append(s, n)
            try:
                slots = bm.append(s, n)
                got = "ok"
                L = m.lens[s]
                pos = np.arange(L - n, L)
                exp = np.array([m.tab[s][p // bs] * bs + p % bs for p in pos], np.int64)
                assert (slots == exp).all()
            except pa.PaError as e:
                got = {pa.PA_ERR_OUT_OF_BLOCKS: "out", pa.PA_ERR_UNSUPPORTED: "unsupported"}[
                    e.status]
            assert got == want
        elif op == "rollback":
            n = int(rng.integers(0, 20))
            want = m.rollback(s, n)
            try:
                bm.rollback(s, n)
                got = "ok"
            except pa.PaError:
                got = "bad"
            assert got == want
        elif op in ("release", "preempt"):
            m.drop(s)
            getattr(bm, op)(s)
        else:
            oldest = m.lens[s]
            want = m.evict(s, oldest)
            assert bm.evict_window(s, oldest).tolist() == want
        tab, lens = check_invariants(bm, ns)
        assert lens.tolist() == m.lens
        assert tab.tolist() == m.tab


def test_prefix_blocks_are_shared_and_reference_counted():
    bm = BlockManager(num_blocks=12, block_size=16, max_seqs=4, max_blocks_per_seq=8)
    bm.append(0, 50)                      # 3 full blocks + 2 tokens
    tab0, _ = bm.tables([0])
    keys = np.array([101, 202, 303], np.uint64)
    with pytest.raises(pa.PaError):
        bm.publish(0, np.array([1, 2, 3, 4], np.uint64))   # block 3 is not full
    bm.publish(0, keys)
    assert bm.stats()["published_blocks"] == 3
    # a request with the same first two blocks, then a different third
    assert bm.attach_prefix(1, np.array([101, 202, 999], np.uint64)) == 2
    tab, lens = check_invariants(bm, 4, shared_ok=True)
    assert lens[1] == 32 and (tab[1, :2] == tab0[0, :2]).all()
    st = bm.stats()
    assert st["shared_blocks"] == 2 and st["prefix_hit_blocks"] == 2
    new = bm.append(1, 5)                 # its own tokens go to a new block
    assert not np.isin(new // 16, tab0[0]).any()
    with pytest.raises(pa.PaError):
        bm.rollback(1, 5 + 3)             # would end inside a shared block
    assert bm.attach_prefix(2, np.array([555], np.uint64)) == 0   # miss
    with pytest.raises(pa.PaError):
        bm.attach_prefix(1, keys)         # only an empty sequence can attach
    free_before = bm.stats()["free_blocks"]
    bm.release(0)                         # the shared blocks stay alive for sequence 1
    st = bm.stats()
    # its third prompt block is cached (keyed, no holder), its partial block freed
    assert st["shared_blocks"] == 0 and st["free_blocks"] == free_before + 1
    assert st["cached_blocks"] == 1
    assert bm.attach_prefix(3, keys) == 3  # two held by sequence 1, one revived
    assert bm.stats()["revived_blocks"] == 1
    bm.release(1)
    bm.release(3)                         # last holders gone: the keyed blocks are cached
    st = bm.stats()
    assert st["free_blocks"] == 9 and st["cached_blocks"] == 3
    assert bm.attach_prefix(2, keys) == 3 and bm.stats()["revived_blocks"] == 4


def test_prefix_outlives_its_request():
    """"llminfer", Prefix KV cache reuse: request r1 runs to completion, then r2
    with the same prompt finds r1's prompt blocks in the prefix cache."""
    bm = BlockManager(num_blocks=20, block_size=16, max_seqs=2, max_blocks_per_seq=8)
    bm.append(0, 40)                      # r1's prompt: 2 full blocks + 8 tokens
    keys = np.array([11, 22], np.uint64)
    bm.publish(0, keys)
    bm.append(0, 5)                       # r1 decodes
    tab1, _ = bm.tables([0])
    bm.release(0)                         # r1 finishes
    st = bm.stats()
    assert st["cached_blocks"] == 2 and st["free_blocks"] == 18 and st["live_seqs"] == 0
    assert bm.attach_prefix(1, keys) == 2  # r2: a hit on both prompt blocks
    tab2, lens2 = check_invariants(bm, 2)
    assert (tab2[1, :2] == tab1[0, :2]).all() and lens2[1] == 32
    st = bm.stats()
    assert st["prefix_hit_blocks"] == 2 and st["revived_blocks"] == 2
    assert st["cached_blocks"] == 0 and st["reclaimed_blocks"] == 0
    new = bm.append(1, 8)                 # r2's own tokens go to a fresh block
    assert not np.isin(new // 16, tab1[0, :2]).any()


def test_prefix_cache_is_reclaimed_under_pressure_lru_first():
    """With no free block left, appends take cached blocks back, least recently
    let go first; a prefix loses its later blocks before its first."""
    bm = BlockManager(num_blocks=8, block_size=4, max_seqs=3, max_blocks_per_seq=10)
    bm.append(0, 12)                      # prompt A: blocks 0, 1, 2
    bm.publish(0, np.array([1, 2, 3], np.uint64))
    bm.append(1, 8)                       # prompt B: blocks 3, 4
    bm.publish(1, np.array([7, 8], np.uint64))
    tab, _ = bm.tables([0, 1])
    bm.release(0)                         # A let go first (least recent), then B
    bm.release(1)
    st = bm.stats()
    assert st["cached_blocks"] == 5 and st["free_blocks"] == 3
    with pytest.raises(pa.PaError) as e:
        bm.append(2, 4 * 9)               # more than free + cached
    assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
    bm.append(2, 4 * 5)                   # 3 free + 2 reclaimed: A's blocks 2, then 1
    st = bm.stats()
    assert st["reclaimed_blocks"] == 2 and st["cached_blocks"] == 3
    t2, _ = bm.tables([2])
    assert set(t2[0, 3:5].tolist()) == {int(tab[0, 2]), int(tab[0, 1])}
    assert bm.attach_prefix(0, np.array([1, 2, 3], np.uint64)) == 1   # only A's head left
    assert bm.attach_prefix(1, np.array([7, 8], np.uint64)) == 2      # B untouched
    check_invariants(bm, 3, shared_ok=True)


class PrefixModel(Model):
    """The header's contract with prefix caching: reference counts, a registry of
    keys and a least-recently-used list of cached blocks."""

    def __init__(self, *a):
        super().__init__(*a)
        self.refs, self.key_of, self.registry, self.lru = {}, {}, {}, []
        self.reclaimed = self.revived = 0

    def pop(self):
        if self.free:
            b = self.free.pop()
        else:
            b = self.lru.pop(0)
            del self.registry[self.key_of.pop(b)]
            self.reclaimed += 1
        self.refs[b] = 1
        return b

    def let_go(self, b):
        self.refs[b] -= 1
        if self.refs[b] == 0:
            (self.lru if b in self.key_of else self.free).append(b)

    def release_range(self, s, lo, hi):
        t = self.tab[s]
        order = [i for i in range(lo, hi) if t[i] >= 0 and not (
            t[i] in self.key_of and self.refs[t[i]] == 1)]
        order += [i for i in range(hi - 1, lo - 1, -1) if t[i] >= 0 and i not in order]
        for i in order:
            self.let_go(t[i])
            t[i] = -1

    def append(self, s, n):
        have, need = self.nblk(self.lens[s]), self.nblk(self.lens[s] + n)
        if need > self.mb:
            return "unsupported"
        if need - have > len(self.free) + len(self.lru):
            return "out"
        for i in range(have, need):
            self.tab[s][i] = self.pop()
        self.lens[s] += n
        return "ok"

    def rollback(self, s, n):
        L2 = self.lens[s] - n
        if n < 0 or L2 < 0 or (self.kept[s] > 0 and L2 - self.w + 1 < self.kept[s] * self.bs):
            return "bad"
        if L2 % self.bs and n > 0:
            b = self.tab[s][L2 // self.bs]
            if b >= 0 and self.refs[b] > 1:
                return "bad"
        self.release_range(s, self.nblk(L2), self.nblk(self.lens[s]))
        self.lens[s] = L2
        return "ok"

    def drop(self, s):
        self.release_range(s, self.kept[s], self.nblk(self.lens[s]))
        self.lens[s], self.kept[s] = 0, 0

    def evict(self, s, oldest):
        if self.w <= 0 or oldest - self.w + 1 <= 0:
            return []
        upto = min((oldest - self.w + 1) // self.bs, self.nblk(self.lens[s]))
        out = []
        for i in range(self.kept[s], upto):
            if self.tab[s][i] >= 0:
                out.append(self.tab[s][i])
                self.let_go(self.tab[s][i])
                self.tab[s][i] = -1
        self.kept[s] = max(self.kept[s], upto)
        return out

    def publish(self, s, keys):
        t = self.tab[s]
        if len(keys) * self.bs > self.lens[s] or any(t[i] < 0 for i in range(len(keys))):
            return "bad"
        for i, k in enumerate(keys):
            if t[i] in self.key_of or k in self.registry:
                continue
            self.registry[k], self.key_of[t[i]] = t[i], k
        return "ok"

    def attach(self, s, keys):
        if self.lens[s] or self.kept[s]:
            return -1
        k = 0
        while k < len(keys) and k < self.mb and keys[k] in self.registry:
            b = self.registry[keys[k]]
            if self.refs[b] == 0:
                self.lru.remove(b)
                self.revived += 1
            self.refs[b] += 1
            self.tab[s][k] = b
            k += 1
        self.lens[s] = k * self.bs
        return k


@pytest.mark.parametrize("seed", range(8))
def test_random_operations_with_prefix_caching_match_the_model(seed):
    """Random appends, rollbacks, releases, preemptions, evictions, publishes and
    prefix attaches, against the model; prompts are drawn from a few shared
    ones, so keys repeat across sequences and cached blocks are revived and
    reclaimed."""
    rng = np.random.default_rng(100 + seed)
    nb, bs, ns, mb, w = 24, int(rng.choice([4, 16])), 5, 10, int(rng.choice([0, 23]))
    bm = BlockManager(nb, bs, ns, mb, w)
    m = PrefixModel(nb, bs, ns, mb, w)
    prompt = [0] * ns   # which shared prompt each sequence's keys come from

    def keys_of(p, n):
        return np.array([1000 * (p + 1) + i for i in range(n)], np.uint64)

    for _ in range(600):
        s = int(rng.integers(ns))
        op = rng.choice(["append", "append", "rollback", "release", "preempt", "evict",
                         "publish", "attach", "attach"])
        if op == "append":
            n = int(rng.integers(0, 20))
            want = m.append(s, n)
            try:
                slots = bm.append(s, n)
                got = "ok"
                L = m.lens[s]
                exp = [m.tab[s][p // bs] * bs + p % bs for p in range(L - n, L)]
                assert slots.tolist() == exp
            except pa.PaError as e:
                got = {pa.PA_ERR_OUT_OF_BLOCKS: "out", pa.PA_ERR_UNSUPPORTED: "unsupported"}[
                    e.status]
            assert got == want
        elif op == "rollback":
            n = int(rng.integers(0, 12))
            want = m.rollback(s, n)
            try:
                bm.rollback(s, n)
                got = "ok"
            except pa.PaError:
                got = "bad"
            assert got == want
        elif op in ("release", "preempt"):
            m.drop(s)
            getattr(bm, op)(s)
        elif op == "evict":
            oldest = m.lens[s]
            want = m.evict(s, oldest)
            assert bm.evict_window(s, oldest).tolist() == want
        elif op == "publish":
            n = int(rng.integers(0, m.lens[s] // bs + 2))
            keys = keys_of(prompt[s], n)
            want = m.publish(s, keys.tolist())
            try:
                bm.publish(s, keys)
                got = "ok"
            except pa.PaError:
                got = "bad"
            assert got == want
        else:
            p = int(rng.integers(3))
            keys = keys_of(p, int(rng.integers(1, mb + 1)))
            want = m.attach(s, keys.tolist())
            try:
                got = bm.attach_prefix(s, keys)
            except pa.PaError:
                got = -1
            assert got == want
            if want >= 0:
                prompt[s] = p
        tab, lens = check_invariants(bm, ns, shared_ok=True)
        assert lens.tolist() == m.lens and tab.tolist() == m.tab
        st = bm.stats()
        assert st["cached_blocks"] == len(m.lru) and st["free_blocks"] == len(m.free)
        assert st["reclaimed_blocks"] == m.reclaimed and st["revived_blocks"] == m.revived

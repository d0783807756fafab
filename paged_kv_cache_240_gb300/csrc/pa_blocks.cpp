// pa_blocks.cpp -- host-side manager of the paged KV cache's physical blocks
// ("PyTorch LLM Serving Engine", What is implemented: fixed-size physical
// blocks, per-sequence block tables, an O(1) free-list allocator, memory
// accounting, recomputation counters after preemption; "MicroGen", Key
// Features: logical-to-physical block mapping, sliding window eviction, KV
// cache state rollback; "Prompt Prefix Caching": token sequence hashing with
// sub-sequence prefix lookup; "llminfer", Architecture: a prefix cache (LRU),
// and its prefix-reuse example, where a finished request's prompt blocks serve
// the next request with the same prompt).  Plain C++ on the host; the C ABI is
// pa_blocks.h.
#include "pa_blocks.h"

#include <algorithm>
#include <new>
#include <unordered_map>
#include <vector>

struct pa_blocks {
  int num_blocks, block_size, max_seqs, max_blocks_per_seq, window;
  std::vector<int32_t> free_stack;  // free block ids; the top is the next allocation
  std::vector<int32_t> tables;      // [max_seqs][max_blocks_per_seq], -1 = no block
  std::vector<int32_t> lens;        // context length per sequence
  std::vector<int32_t> first_kept;  // logical blocks below this were evicted
  std::vector<int32_t> refs;        // sequences holding each block
  std::vector<uint64_t> key_of;     // the prefix key a block is registered under
  std::vector<uint8_t> keyed;       // whether it is registered
  std::unordered_map<uint64_t, int32_t> registry;  // prefix key -> block
  // The prefix cache: registered blocks that no sequence holds any more keep
  // their K/V and their key, on a list ordered by when they were let go (least
  // recently used at the head).  An allocation takes a free block first, and
  // reclaims the head of this list only when none is left.
  std::vector<int32_t> lru_prev, lru_next;  // intrusive list links, -1 = none
  int32_t lru_head = -1, lru_tail = -1;
  int cached = 0;
  pa_blocks_stats stats;

  int32_t* table(int seq) { return tables.data() + (size_t)seq * max_blocks_per_seq; }
  const int32_t* table(int seq) const {
    return tables.data() + (size_t)seq * max_blocks_per_seq;
  }
  bool valid_seq(int seq) const { return seq >= 0 && seq < max_seqs; }
  int blocks_for(long long tokens) const {
    return (int)((tokens + block_size - 1) / block_size);
  }
  // Blocks an allocation can take: free ones and cached ones.
  long long available() const { return (long long)free_stack.size() + cached; }

  void lru_push_back(int32_t b) {  // b becomes the most recently used
    lru_prev[b] = lru_tail;
    lru_next[b] = -1;
    if (lru_tail >= 0) lru_next[lru_tail] = b;
    else lru_head = b;
    lru_tail = b;
    cached++;
  }
  void lru_remove(int32_t b) {
    if (lru_prev[b] >= 0) lru_next[lru_prev[b]] = lru_next[b];
    else lru_head = lru_next[b];
    if (lru_next[b] >= 0) lru_prev[lru_next[b]] = lru_prev[b];
    else lru_tail = lru_prev[b];
    lru_prev[b] = lru_next[b] = -1;
    cached--;
  }
  // A block for a new position: the top of the free list, else the least
  // recently used cached block, whose key is dropped.  The caller has checked
  // available() > 0.
  int32_t pop_free() {
    int32_t b;
    if (!free_stack.empty()) {
      b = free_stack.back();
      free_stack.pop_back();
    } else {
      b = lru_head;
      lru_remove(b);
      registry.erase(key_of[b]);
      keyed[b] = 0;
      stats.reclaimed_blocks++;
    }
    refs[b] = 1;
    return b;
  }
  // One holder lets block b go.  The last one returns it to the free list, or,
  // if it is registered under a prefix key, to the tail of the prefix cache.
  void push_free(int32_t b) {
    if (--refs[b] > 0) {
      if (refs[b] == 1) stats.shared_blocks--;
      return;
    }
    if (keyed[b]) lru_push_back(b);
    else free_stack.push_back(b);
  }
  // Return logical blocks [from, to) of seq (skipping holes).  Unregistered
  // blocks go to the free list in table order; registered ones go to the cache
  // last block first, so that a prefix's later blocks are reclaimed before its
  // earlier ones (a prefix is found from its first block on).
  void free_range(int seq, int from, int to) {
    int32_t* t = table(seq);
    for (int i = from; i < to; i++)
      if (t[i] >= 0 && !(keyed[t[i]] && refs[t[i]] == 1)) {
        push_free(t[i]);
        t[i] = -1;
      }
    for (int i = to - 1; i >= from; i--)
      if (t[i] >= 0) {
        push_free(t[i]);
        t[i] = -1;
      }
  }
  void drop_all(int seq) {
    free_range(seq, first_kept[seq], blocks_for(lens[seq]));
    stats.tokens_held -= lens[seq];
    if (lens[seq] > 0) stats.live_seqs--;
    lens[seq] = 0;
    first_kept[seq] = 0;
  }
};

extern "C" pa_blocks* pa_blocks_create(int num_blocks, int block_size, int max_seqs,
                                       int max_blocks_per_seq, int window) {
  if (num_blocks < 1 || block_size < 1 || max_seqs < 1 || max_blocks_per_seq < 1 || window < 0)
    return nullptr;
  if ((long long)max_blocks_per_seq * block_size > 0x7fffffffLL ||
      (long long)num_blocks * block_size > 0x7fffffffLL)
    return nullptr;
  pa_blocks* bm = new (std::nothrow) pa_blocks;
  if (!bm) return nullptr;
  try {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->max_seqs = max_seqs;
    bm->max_blocks_per_seq = max_blocks_per_seq;
    bm->window = window;
    bm->free_stack.reserve(num_blocks);
    // lowest ids on top, so a fresh pool hands out 0, 1, 2, ...
    for (int b = num_blocks - 1; b >= 0; b--) bm->free_stack.push_back(b);
    bm->tables.assign((size_t)max_seqs * max_blocks_per_seq, -1);
    bm->lens.assign(max_seqs, 0);
    bm->first_kept.assign(max_seqs, 0);
    bm->refs.assign(num_blocks, 0);
    bm->key_of.assign(num_blocks, 0);
    bm->keyed.assign(num_blocks, 0);
    bm->lru_prev.assign(num_blocks, -1);
    bm->lru_next.assign(num_blocks, -1);
  } catch (...) {
    delete bm;
    return nullptr;
  }
  bm->stats = pa_blocks_stats{};
  bm->stats.num_blocks = num_blocks;
  return bm;
}

extern "C" void pa_blocks_destroy(pa_blocks* bm) { delete bm; }

extern "C" pa_status pa_blocks_append(pa_blocks* bm, int seq, int num_tokens,
                                      int32_t* slots_out) {
  if (!bm || !bm->valid_seq(seq) || num_tokens < 0 || (num_tokens > 0 && !slots_out))
    return PA_ERR_INVALID_ARG;
  const long long L = bm->lens[seq], L2 = L + num_tokens;
  const int have = bm->blocks_for(L), need = bm->blocks_for(L2);
  if (need > bm->max_blocks_per_seq) return PA_ERR_UNSUPPORTED;
  if (need - have > bm->available()) return PA_ERR_OUT_OF_BLOCKS;
  int32_t* t = bm->table(seq);
  for (int i = have; i < need; i++) t[i] = bm->pop_free();
  for (int k = 0; k < num_tokens; k++) {
    const long long p = L + k;
    slots_out[k] = (int32_t)(t[p / bm->block_size] * (long long)bm->block_size +
                             p % bm->block_size);
  }
  if (L == 0 && num_tokens > 0) bm->stats.live_seqs++;
  bm->lens[seq] = (int32_t)L2;
  bm->stats.tokens_held += num_tokens;
  return PA_OK;
}

extern "C" pa_status pa_blocks_rollback(pa_blocks* bm, int seq, int num_tokens) {
  if (!bm || !bm->valid_seq(seq) || num_tokens < 0 || num_tokens > bm->lens[seq])
    return PA_ERR_INVALID_ARG;
  const int L2 = bm->lens[seq] - num_tokens;
  // after an eviction, the next query (at position L2) must still find every key
  // of its window in a kept block
  if (bm->first_kept[seq] > 0 &&
      (long long)L2 - bm->window + 1 < (long long)bm->first_kept[seq] * bm->block_size)
    return PA_ERR_INVALID_ARG;
  // the next append would write into the block holding position L2
  if (L2 % bm->block_size != 0 && num_tokens > 0) {
    const int32_t b = bm->table(seq)[L2 / bm->block_size];
    if (b >= 0 && bm->refs[b] > 1) return PA_ERR_INVALID_ARG;
  }
  bm->free_range(seq, bm->blocks_for(L2), bm->blocks_for(bm->lens[seq]));
  if (L2 == 0 && num_tokens > 0) bm->stats.live_seqs--;
  bm->lens[seq] = L2;
  bm->stats.tokens_held -= num_tokens;
  bm->stats.rolled_back_tokens += num_tokens;
  return PA_OK;
}

extern "C" pa_status pa_blocks_release(pa_blocks* bm, int seq) {
  if (!bm || !bm->valid_seq(seq)) return PA_ERR_INVALID_ARG;
  bm->drop_all(seq);
  return PA_OK;
}

extern "C" pa_status pa_blocks_preempt(pa_blocks* bm, int seq) {
  if (!bm || !bm->valid_seq(seq)) return PA_ERR_INVALID_ARG;
  if (bm->lens[seq] > 0) {
    bm->stats.preemptions++;
    bm->stats.recompute_tokens += bm->lens[seq];
  }
  bm->drop_all(seq);
  return PA_OK;
}

extern "C" int pa_blocks_evict_window(pa_blocks* bm, int seq, int oldest_query,
                                      int32_t* freed_out, int cap) {
  if (!bm || !bm->valid_seq(seq) || cap < 0 || oldest_query < 0) return -1;
  if (bm->window <= 0) return 0;
  // the earliest key any query at oldest_query or later can see
  const long long lo = (long long)oldest_query - bm->window + 1;
  if (lo <= 0) return 0;
  // blocks whose last position is below lo, and that hold positions at all
  const int upto = (int)std::min<long long>(lo / bm->block_size, bm->blocks_for(bm->lens[seq]));
  int32_t* t = bm->table(seq);
  int freed = 0;
  for (int i = bm->first_kept[seq]; i < upto; i++) {
    if (t[i] < 0) continue;
    if (freed_out && freed < cap) freed_out[freed] = t[i];
    freed++;
    bm->push_free(t[i]);
    t[i] = -1;
  }
  bm->first_kept[seq] = std::max(bm->first_kept[seq], upto);
  bm->stats.evicted_blocks += freed;
  return freed;
}

extern "C" pa_status pa_blocks_tables(const pa_blocks* bm, const int32_t* seqs, int n,
                                      int32_t* tables_out, int32_t* context_lens_out) {
  if (!bm || n < 0 || (n > 0 && !seqs)) return PA_ERR_INVALID_ARG;
  for (int i = 0; i < n; i++)
    if (!bm->valid_seq(seqs[i])) return PA_ERR_INVALID_ARG;
  for (int i = 0; i < n; i++) {
    if (tables_out)
      std::copy(bm->table(seqs[i]), bm->table(seqs[i]) + bm->max_blocks_per_seq,
                tables_out + (size_t)i * bm->max_blocks_per_seq);
    if (context_lens_out) context_lens_out[i] = bm->lens[seqs[i]];
  }
  return PA_OK;
}

extern "C" pa_status pa_blocks_publish(pa_blocks* bm, int seq, const uint64_t* keys,
                                       int n_blocks) {
  if (!bm || !bm->valid_seq(seq) || n_blocks < 0 || (n_blocks > 0 && !keys))
    return PA_ERR_INVALID_ARG;
  if ((long long)n_blocks * bm->block_size > bm->lens[seq] || n_blocks > bm->max_blocks_per_seq)
    return PA_ERR_INVALID_ARG;
  const int32_t* t = bm->table(seq);
  for (int i = 0; i < n_blocks; i++)
    if (t[i] < 0) return PA_ERR_INVALID_ARG;  // evicted
  try {
    for (int i = 0; i < n_blocks; i++) {
      const int32_t b = t[i];
      if (bm->keyed[b] || bm->registry.count(keys[i])) continue;
      bm->registry.emplace(keys[i], b);
      bm->key_of[b] = keys[i];
      bm->keyed[b] = 1;
      bm->stats.published_blocks++;
    }
  } catch (...) {
    return PA_ERR_INVALID_ARG;  // out of host memory: the registry keeps what it has
  }
  return PA_OK;
}

extern "C" int pa_blocks_attach_prefix(pa_blocks* bm, int seq, const uint64_t* keys,
                                       int n_blocks) {
  if (!bm || !bm->valid_seq(seq) || n_blocks < 0 || (n_blocks > 0 && !keys)) return -1;
  if (bm->lens[seq] != 0 || bm->first_kept[seq] != 0) return -1;
  int32_t* t = bm->table(seq);
  int k = 0;
  for (; k < n_blocks && k < bm->max_blocks_per_seq; k++) {
    const auto hit = bm->registry.find(keys[k]);
    if (hit == bm->registry.end()) break;
    const int32_t b = hit->second;
    if (bm->refs[b] == 0) {  // in the prefix cache: revived
      bm->lru_remove(b);
      bm->stats.revived_blocks++;
    }
    if (++bm->refs[b] == 2) bm->stats.shared_blocks++;
    t[k] = b;
  }
  if (k > 0) {
    bm->lens[seq] = k * bm->block_size;
    bm->stats.live_seqs++;
    bm->stats.tokens_held += (long long)k * bm->block_size;
    bm->stats.prefix_hit_blocks += k;
  }
  return k;
}

extern "C" int pa_blocks_context_len(const pa_blocks* bm, int seq) {
  if (!bm || !bm->valid_seq(seq)) return -1;
  return bm->lens[seq];
}

extern "C" pa_status pa_blocks_get_stats(const pa_blocks* bm, pa_blocks_stats* out) {
  if (!bm || !out) return PA_ERR_INVALID_ARG;
  *out = bm->stats;
  out->free_blocks = (int)bm->free_stack.size();
  out->cached_blocks = bm->cached;
  return PA_OK;
}
